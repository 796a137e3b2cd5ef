"""Host-only checks of the C ABI: the library loads, exports every declared entry point, and
rejects bad arguments with the documented status before touching the GPU."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

from gaussian_mixture_sequence_gma_gb300 import build as gbuild
from gaussian_mixture_sequence_gma_gb300 import gma

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include"))) if f.endswith(".h")]


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gma.lib()


def declared_symbols():
    names = []
    for h in HEADERS:
        src = open(h).read()
        names += re.findall(r"GMA_API\s+[\w\s\*]+?\b(gma_\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert set(gma.EXPORTED) <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", gma.lib_path()], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(gma_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(L, n)


def test_status_strings_and_version(L):
    for s in range(7):
        assert len(gma.status_string(s)) > 0
    assert L.gma_version() >= 1


def P(**kw):
    base = dict(B=1, H=2, N=256, K=16, dtype=gma.GMA_BF16, eps=1e-6, d=64, dv=64)
    base.update(kw)
    return gma.problem(base["B"], base["H"], base["N"], base["K"], base["dtype"], base["eps"], base["d"], base["dv"])


def test_workspace_bytes(L):
    for op in (gma.OP_RESPONSIBILITIES, gma.OP_BIDIR, gma.OP_CAUSAL):
        for dt in (gma.GMA_F32, gma.GMA_BF16):
            assert gma.workspace_bytes(P(dtype=dt), op) > 0
            assert gma.workspace_bytes(P(dtype=dt), op) % 256 == 0
    assert gma.workspace_bytes(P(d=32), gma.OP_BIDIR) == 0
    assert gma.workspace_bytes(P(K=257), gma.OP_BIDIR) == 0
    assert gma.workspace_bytes(P(B=0), gma.OP_BIDIR) == 0
    assert gma.workspace_bytes(P(dtype=7), gma.OP_BIDIR) == 0
    assert gma.workspace_bytes(P(), 10) == 0
    # workspace does not grow with N for the bidirectional write state beyond the fixed split
    assert gma.workspace_bytes(P(N=1 << 20), gma.OP_BIDIR) == gma.workspace_bytes(P(N=1 << 16), gma.OP_BIDIR)


def _segments(BH, tiles, sms=152):
    """The causal path's segment count per head row: over the largest count fitting in w = 1..8 waves of
    one CTA per SM, the one with the fewest waves * (tiles per segment + 1); ties to fewer segments."""
    best, best_cost = 1, None
    for w in range(1, 9):
        s = max(1, min(w * sms // BH, tiles))
        seg = -(-tiles // s)
        splits = -(-tiles // seg)
        cost = -(-BH * splits // sms) * (seg + 1)
        if best_cost is None or cost < best_cost or (cost == best_cost and splits < best):
            best, best_cost = splits, cost
    return best


@pytest.mark.parametrize("B,H,N,K,want", [(8, 12, 2048, 256, 3), (4, 8, 4096, 128, 4), (1, 8, 131072, 256, 19),
                                          (12, 1, 8192, 64, 11), (1000, 1, 2048, 256, 1)])
def test_causal_segments_follow_the_wave_rule(B, H, N, K, want):
    """bf16 causal workspace = a part independent of N + B*H segments x Kp x 80 float32 aggregates, so
    the difference against a one-tile problem (one segment) gives the segment count the library chose."""
    kp = 64 if K <= 64 else (128 if K <= 128 else 256)
    assert _segments(B * H, N // 128) == want
    big = gma.workspace_bytes(P(B=B, H=H, N=N, K=K), gma.OP_CAUSAL)
    one = gma.workspace_bytes(P(B=B, H=H, N=128, K=K), gma.OP_CAUSAL)
    per_segment = B * H * kp * 80 * 4
    # both totals are rounded up to 256 bytes; the aggregates are a multiple of 256 bytes here
    assert big - one == (want - 1) * per_segment


# Fake, 256-aligned "device" addresses: every call below must fail (or no-op) before any CUDA call.
A = 1 << 20


def call(L, name, prob, ptrs=None, ws_bytes=1 << 30):
    p = [A + i * (1 << 16) for i in range(8)] if ptrs is None else ptrs
    if name == "gma_responsibilities":
        return L.gma_responsibilities(ctypes.byref(prob), p[0], p[3], p[4], p[5], p[6], p[7], ws_bytes, None)
    return getattr(L, name)(ctypes.byref(prob), p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], ws_bytes, None)


@pytest.mark.parametrize("name", ["gma_responsibilities", "gma_forward_bidir", "gma_forward_causal"])
def test_argument_errors(L, name):
    assert call(L, name, P(d=32)) == gma.GMA_ERR_UNSUPPORTED
    assert call(L, name, P(dv=128)) == gma.GMA_ERR_UNSUPPORTED
    assert call(L, name, P(K=300)) == gma.GMA_ERR_UNSUPPORTED
    assert call(L, name, P(dtype=5)) == gma.GMA_ERR_UNSUPPORTED
    assert call(L, name, P(B=0)) == gma.GMA_ERR_INVALID_ARG
    assert call(L, name, P(K=0)) == gma.GMA_ERR_INVALID_ARG
    assert call(L, name, P(N=-1)) == gma.GMA_ERR_INVALID_ARG
    assert call(L, name, P(eps=-1.0)) == gma.GMA_ERR_INVALID_ARG
    assert call(L, name, P(eps=float("nan"))) == gma.GMA_ERR_INVALID_ARG
    assert call(L, name, P(B=1 << 16, H=1 << 8, N=1 << 8)) == gma.GMA_ERR_UNSUPPORTED
    ptrs = [A + i * (1 << 16) for i in range(8)]
    for i in (0, 3, 4, 5, 6, 7):
        bad = list(ptrs); bad[i] = None
        assert call(L, name, P(), bad) == gma.GMA_ERR_INVALID_ARG
    for i in (0, 3, 4, 5, 6):
        bad = list(ptrs); bad[i] += 2
        assert call(L, name, P(), bad) == gma.GMA_ERR_INVALID_ARG
    bad = list(ptrs); bad[7] += 16  # workspace must be 256-aligned
    assert call(L, name, P(), bad) == gma.GMA_ERR_INVALID_ARG
    op = {"gma_responsibilities": 0, "gma_forward_bidir": 1, "gma_forward_causal": 2}[name]
    need = gma.workspace_bytes(P(), op)
    assert call(L, name, P(), ws_bytes=need - 1) == gma.GMA_ERR_WORKSPACE
    # N == 0 is a no-op that launches nothing; the (empty) tensors may then be null
    assert call(L, name, P(N=0), ws_bytes=gma.workspace_bytes(P(N=0), op)) == gma.GMA_OK
    nul = [None, None, None, A + 3 * (1 << 16), A + 4 * (1 << 16), A + 5 * (1 << 16), None, A + 7 * (1 << 16)]
    assert call(L, name, P(N=0), nul, ws_bytes=gma.workspace_bytes(P(N=0), op)) == gma.GMA_OK


@pytest.mark.parametrize("name", ["gma_forward_bidir", "gma_forward_causal"])
def test_forward_specific_errors(L, name):
    ptrs = [A + i * (1 << 16) for i in range(8)]
    for i in (1, 2):
        bad = list(ptrs); bad[i] = None
        assert call(L, name, P(), bad) == gma.GMA_ERR_INVALID_ARG
        bad = list(ptrs); bad[i] += 8
        assert call(L, name, P(), bad) == gma.GMA_ERR_INVALID_ARG
    for i in (0, 1, 2):  # output aliasing an input
        bad = list(ptrs); bad[6] = bad[i]
        assert call(L, name, P(), bad) == gma.GMA_ERR_INVALID_ARG


def call_cross(L, prob, Nk, ptrs=None, ws_bytes=1 << 30):
    p = [A + i * (1 << 16) for i in range(8)] if ptrs is None else ptrs
    return L.gma_forward_cross(ctypes.byref(prob), Nk, p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], ws_bytes, None)


def test_cross_argument_errors(L):
    for dt in (gma.GMA_F32, gma.GMA_BF16):
        assert gma.workspace_bytes(P(dtype=dt), gma.OP_CROSS) == gma.workspace_bytes(P(dtype=dt), gma.OP_BIDIR)
    assert call_cross(L, P(), -1) == gma.GMA_ERR_INVALID_ARG
    assert call_cross(L, P(d=32), 16) == gma.GMA_ERR_UNSUPPORTED
    assert call_cross(L, P(B=1 << 8, H=1 << 8), 1 << 15) == gma.GMA_ERR_UNSUPPORTED
    ptrs = [A + i * (1 << 16) for i in range(8)]
    for i in (1, 2):  # K / V needed when Nk > 0
        bad = list(ptrs); bad[i] = None
        assert call_cross(L, P(), 7, bad) == gma.GMA_ERR_INVALID_ARG
        bad = list(ptrs); bad[i] += 8
        assert call_cross(L, P(), 7, bad) == gma.GMA_ERR_INVALID_ARG
    for i in (0, 1, 2):
        bad = list(ptrs); bad[6] = bad[i]
        assert call_cross(L, P(), 7, bad) == gma.GMA_ERR_INVALID_ARG
    need = gma.workspace_bytes(P(), gma.OP_CROSS)
    assert call_cross(L, P(), 7, ws_bytes=need - 1) == gma.GMA_ERR_WORKSPACE
    # no queries: a no-op, every tensor may be null
    nul = [None, None, None, A + 3 * (1 << 16), A + 4 * (1 << 16), A + 5 * (1 << 16), None, A + 7 * (1 << 16)]
    assert call_cross(L, P(N=0), 5, nul, ws_bytes=need) == gma.GMA_OK


def test_state_and_decode_argument_errors(L):
    assert L.gma_state_bytes(ctypes.byref(P(B=2, H=3, K=17))) == 2 * 3 * 17 * 65 * 4
    assert L.gma_state_bytes(ctypes.byref(P(d=32))) == 0
    for op in (gma.OP_CAUSAL_STATE, gma.OP_CAUSAL_DECODE):
        for dt in (gma.GMA_F32, gma.GMA_BF16):
            n = gma.workspace_bytes(P(dtype=dt), op)
            assert n > 0 and n % 256 == 0
    assert gma.workspace_bytes(P(), 10) == 0
    ptr = [A + i * (1 << 16) for i in range(10)]

    def st(prob, p=ptr, ws_bytes=1 << 30):  # K, V, mu, sigma2, log_pi, state, ws
        return L.gma_causal_state(ctypes.byref(prob), p[1], p[2], p[3], p[4], p[5], p[8], p[7], ws_bytes, None)

    def dec(prob, p=ptr, ws_bytes=1 << 30):  # Q, K, V, mu, sigma2, log_pi, state, O, ws
        return L.gma_causal_decode(ctypes.byref(prob), p[0], p[1], p[2], p[3], p[4], p[5], p[8], p[6], p[7],
                                   ws_bytes, None)

    for f in (st, dec):
        assert f(P(d=32)) == gma.GMA_ERR_UNSUPPORTED
        assert f(P(K=0)) == gma.GMA_ERR_INVALID_ARG
        for i in (1, 2, 3, 8):
            bad = list(ptr); bad[i] = None
            assert f(P(), bad) == gma.GMA_ERR_INVALID_ARG
            bad = list(ptr); bad[i] += 4
            assert f(P(), bad) == gma.GMA_ERR_INVALID_ARG
        bad = list(ptr); bad[7] += 16
        assert f(P(), bad) == gma.GMA_ERR_INVALID_ARG
    assert st(P(), ws_bytes=gma.workspace_bytes(P(), gma.OP_CAUSAL_STATE) - 1) == gma.GMA_ERR_WORKSPACE
    assert dec(P(), ws_bytes=gma.workspace_bytes(P(), gma.OP_CAUSAL_DECODE) - 1) == gma.GMA_ERR_WORKSPACE
    for i in (0, 1, 2, 8):  # output aliasing an input or the state
        bad = list(ptr); bad[6] = bad[i]
        assert dec(P(), bad) == gma.GMA_ERR_INVALID_ARG
    # no new tokens: a no-op; Q, K, V and O may be null
    nul = [None, None, None] + ptr[3:6] + [None] + ptr[7:]
    assert dec(P(N=0), nul) == gma.GMA_OK


@pytest.mark.parametrize("name,op", [("gma_backward_bidir", 6), ("gma_backward_causal", 7)])
def test_backward_argument_errors(L, name, op):
    for dt in (gma.GMA_F32, gma.GMA_BF16):
        n1 = gma.workspace_bytes(P(dtype=dt, N=256), op)
        n2 = gma.workspace_bytes(P(dtype=dt, N=512), op)
        assert n1 > 0 and n1 % 256 == 0 and n2 > n1  # holds the per-row softmax gradients
    ptr = [A + i * (1 << 16) for i in range(16)]

    def bwd(prob, p=ptr, ws_bytes=1 << 30):  # Q K V mu s2 lp dO | dQ dK dV dmu ds2 dlp | ws
        return getattr(L, name)(ctypes.byref(prob), *p[0:13], p[13], ws_bytes, None)

    assert bwd(P(d=32)) == gma.GMA_ERR_UNSUPPORTED
    assert bwd(P(K=0)) == gma.GMA_ERR_INVALID_ARG
    for i in range(13):
        bad = list(ptr); bad[i] = None
        assert bwd(P(), bad) == gma.GMA_ERR_INVALID_ARG, i
        bad = list(ptr); bad[i] += 4
        assert bwd(P(), bad) == gma.GMA_ERR_INVALID_ARG, i
    for o in range(7, 13):  # an output aliasing an input or another output
        for i in range(13):
            if i == o:
                continue
            bad = list(ptr); bad[o] = bad[i]
            assert bwd(P(), bad) == gma.GMA_ERR_INVALID_ARG, (o, i)
    bad = list(ptr); bad[13] += 16
    assert bwd(P(), bad) == gma.GMA_ERR_INVALID_ARG
    assert bwd(P(), ws_bytes=gma.workspace_bytes(P(), op) - 1) == gma.GMA_ERR_WORKSPACE


def test_check_device_error_rejects_bad_workspace(L):
    assert L.gma_check_device_error(None, None) == gma.GMA_ERR_INVALID_ARG
    assert L.gma_check_device_error(A + 16, None) == gma.GMA_ERR_INVALID_ARG


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "gaussian_mixture_sequence_gma_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, re.M), f
                assert "gma_oracle" not in src and "liboracle" not in src, f


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(gma, "_lib", None)
    monkeypatch.setattr(gma, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        gma.lib()


def test_projected_argument_errors(L):
    for dt in (gma.GMA_F32, gma.GMA_BF16):
        for op, base in ((gma.OP_PROJECTED_BIDIR, gma.OP_BIDIR), (gma.OP_PROJECTED_CAUSAL, gma.OP_CAUSAL)):
            n = gma.workspace_bytes(P(dtype=dt), op)
            pr = P(dtype=dt)
            qkv = 3 * (-(-pr.B * pr.H * pr.N * 64 * (2 if dt == gma.GMA_BF16 else 4) // 256) * 256)
            fwd = -(-gma.workspace_bytes(pr, base) // 256) * 256
            if dt == gma.GMA_BF16:
                # the forward's own workspace and Q, K, V (the tcgen05 projection keeps no float32 Y)
                assert n == fwd + qkv
            else:
                # the forward's own workspace, the library GEMM's, Y float32 [B*N][3*H*64] and Q, K, V
                assert n % 256 == 0 and n > fwd + 32 * (1 << 20) + 256 * 384 * 4 + qkv - 256
    ptr = [A + i * (1 << 16) for i in range(10)]

    def proj(prob, causal=1, dm=128, p=ptr, ws_bytes=1 << 34):  # X W b mu s2 lp O ws
        return L.gma_forward_projected(ctypes.byref(prob), causal, dm, p[0], p[1], p[2], p[3], p[4], p[5], p[6],
                                       p[7], ws_bytes, None)

    assert proj(P(d=32)) == gma.GMA_ERR_UNSUPPORTED
    assert proj(P(), causal=2) == gma.GMA_ERR_INVALID_ARG
    for dm in (0, 4, 100):
        assert proj(P(), dm=dm) == gma.GMA_ERR_UNSUPPORTED
    for i in range(8):
        bad = list(ptr); bad[i] = None
        assert proj(P(), p=bad) == gma.GMA_ERR_INVALID_ARG
    for i in range(7):
        bad = list(ptr); bad[i] += 4
        assert proj(P(), p=bad) == gma.GMA_ERR_INVALID_ARG
    for i in (0, 1, 2):  # output aliasing an input
        bad = list(ptr); bad[6] = bad[i]
        assert proj(P(), p=bad) == gma.GMA_ERR_INVALID_ARG
    need = gma.workspace_bytes(P(), gma.OP_PROJECTED_CAUSAL)
    assert proj(P(), ws_bytes=need - 1) == gma.GMA_ERR_WORKSPACE
    nul = [None, ptr[1], ptr[2], ptr[3], ptr[4], ptr[5], None, ptr[7]]
    assert proj(P(N=0), p=nul, ws_bytes=gma.workspace_bytes(P(N=0), gma.OP_PROJECTED_CAUSAL)) == gma.GMA_OK


def test_prepared_decode_argument_errors(L):
    """gma_decode_prepare / gma_causal_decode_prepared check their arguments before any CUDA call."""
    ptr = [A + i * (1 << 16) for i in range(10)]
    need = gma.workspace_bytes(P(), gma.OP_CAUSAL_DECODE)

    def prep(prob, p=ptr, ws_bytes=1 << 30):  # mu, sigma2, log_pi, ws
        return L.gma_decode_prepare(ctypes.byref(prob), p[3], p[4], p[5], p[7], ws_bytes, None)

    def run(prob, p=ptr, ws_bytes=1 << 30):  # Q, K, V, state, O, ws
        return L.gma_causal_decode_prepared(ctypes.byref(prob), p[0], p[1], p[2], p[8], p[6], p[7], ws_bytes, None)

    for f, idx in ((prep, (3, 4, 5, 7)), (run, (0, 1, 2, 6, 7, 8))):
        assert f(P(d=32)) == gma.GMA_ERR_UNSUPPORTED
        assert f(P(K=0)) == gma.GMA_ERR_INVALID_ARG
        assert f(P(K=300)) == gma.GMA_ERR_UNSUPPORTED
        for i in idx:
            bad = list(ptr)
            bad[i] = None
            assert f(P(), bad) == gma.GMA_ERR_INVALID_ARG, (f.__name__, i)
            bad[i] = ptr[i] + 4
            assert f(P(), bad) == gma.GMA_ERR_INVALID_ARG, (f.__name__, i)
        assert f(P(), ws_bytes=need - 1) == gma.GMA_ERR_WORKSPACE
    # outputs may not alias an input or the state
    for j in (0, 1, 2, 8):
        alias = list(ptr)
        alias[6] = ptr[j]
        assert run(P(), alias) == gma.GMA_ERR_INVALID_ARG
    # no new token: nothing to do, also without Q, K, V and O
    assert run(P(N=0), [None, None, None, None, None, None, None, ptr[7], ptr[8], None], ws_bytes=need) == gma.GMA_OK


def test_decode_workspace_size():
    """The decode workspace is the documented control block (256 B) plus every head's folded parameters,
    4 H (128 (K + 1) + K) bytes with each head's block rounded up to 16 bytes, the total to 256."""
    for B, H, K in ((1, 1, 1), (2, 3, 17), (8, 12, 256), (4, 8, 128)):
        head = (2 * 64 * (K + 1) + K + 3) // 4 * 4 * 4
        want = 256 + (H * head + 255) // 256 * 256
        for dt in (gma.GMA_F32, gma.GMA_BF16):
            for N in (1, 64):
                assert gma.workspace_bytes(P(B=B, H=H, K=K, N=N, dtype=dt), gma.OP_CAUSAL_DECODE) == want


def test_static_ws_binding_rejects_mixed_dtypes_before_any_call(L, monkeypatch):
    """forward_bidir_static_ws checks that K and V share Q's dtype (the library reads them with Q's
    element size) and that a caller-supplied out matches Q, before anything reaches the library."""
    import torch

    def never(*a, **k):
        raise AssertionError("the library must not be called")

    monkeypatch.setattr(gma, "_check_cuda", never)
    q = torch.zeros(1, 2, 8, 64, dtype=torch.float32)
    kb = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    mu, s2, lp = torch.zeros(2, 4, 64), torch.ones(2, 4, 64), torch.zeros(2, 4)
    with pytest.raises(TypeError):
        gma.forward_bidir_static_ws(q, kb, q, mu, s2, lp)
    with pytest.raises(TypeError):
        gma.forward_bidir_static_ws(q, q, kb, mu, s2, lp)
    with pytest.raises(TypeError):
        gma.forward_bidir_static_ws(q, q, q, mu, s2, lp, out=torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        gma.forward_bidir_static_ws(q, q, q, mu, s2, lp, out=torch.zeros(1, 2, 7, 64))
    with pytest.raises(ValueError):
        gma.forward_bidir_static_ws(q, torch.zeros(1, 2, 9, 64), q, mu, s2, lp)


def test_wait_limit_setter(L):
    """The bounded-wait limit: default 1 s, settable within [1 ms, 10 min], 0 restores the default,
    out-of-range values are refused and leave the limit unchanged."""
    assert L.gma_set_wait_limit_ns(0) == gma.GMA_OK
    default = L.gma_get_wait_limit_ns()
    env = os.environ.get("GMA_WAIT_LIMIT_MS")
    assert default == (int(float(env) * 1e6) if env else 1_000_000_000)
    try:
        assert L.gma_set_wait_limit_ns(20_000_000) == gma.GMA_OK
        assert L.gma_get_wait_limit_ns() == 20_000_000
        assert L.gma_set_wait_limit_ns(999_999) == gma.GMA_ERR_INVALID_ARG
        assert L.gma_set_wait_limit_ns(600_000_000_001) == gma.GMA_ERR_INVALID_ARG
        assert L.gma_get_wait_limit_ns() == 20_000_000
        gma.set_wait_limit_ns(5_000_000)
        assert gma.wait_limit_ns() == 5_000_000
        with pytest.raises(gma.GmaError):
            gma.set_wait_limit_ns(1)
    finally:
        assert L.gma_set_wait_limit_ns(0) == gma.GMA_OK
    assert L.gma_get_wait_limit_ns() == default


def test_wait_limit_environment_variable():
    """GMA_WAIT_LIMIT_MS sets the default of a fresh process (clamped to [1 ms, 10 min])."""
    code = ("from gaussian_mixture_sequence_gma_gb300 import gma; print(gma.wait_limit_ns())")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for ms, want in (("250", 250_000_000), ("0.0001", 1_000_000), ("1e9", 600_000_000_000), ("junk", 1_000_000_000)):
        env = dict(os.environ, GMA_WAIT_LIMIT_MS=ms)
        out = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True,
                             timeout=120)
        assert out.returncode == 0, out.stderr
        assert int(out.stdout.strip().splitlines()[-1]) == want, ms


def _align(x, a=256):
    return -(-x // a) * a


def test_deterministic_mode_setter_and_workspace(L):
    """The deterministic reduction mode: 1 / 0 / -1 (the default), others refused; with it on, the
    workspaces of the calls whose sums cross CTAs grow by their documented partials and the others
    do not change."""
    assert L.gma_set_deterministic(-1) == gma.GMA_OK
    default = L.gma_get_deterministic()
    env = os.environ.get("GMA_DETERMINISTIC", "")
    assert default == (1 if env not in ("", "0") else 0)
    try:
        assert L.gma_set_deterministic(0) == gma.GMA_OK
        off = {(op, dt): gma.workspace_bytes(P(B=2, H=3, N=4096, K=100, dtype=dt), op)
               for op in range(9) for dt in (gma.GMA_F32, gma.GMA_BF16)}
        assert L.gma_set_deterministic(1) == gma.GMA_OK
        assert L.gma_get_deterministic() == 1 and gma.deterministic()
        on = {(op, dt): gma.workspace_bytes(P(B=2, H=3, N=4096, K=100, dtype=dt), op)
              for op in range(9) for dt in (gma.GMA_F32, gma.GMA_BF16)}
        BH, K, kp = 6, 100, 128
        for op in (gma.OP_BIDIR, gma.OP_CROSS, gma.OP_CAUSAL_STATE):
            # bf16: one 80-column state per write CTA, at most max(152, B*H) CTAs
            assert on[op, gma.GMA_BF16] == _align(off[op, gma.GMA_BF16]) + _align(max(152, BH) * kp * 80 * 4)
            # float32: one 65-column state per write CTA, at most 304 + B*H CTAs
            assert on[op, gma.GMA_F32] == _align(off[op, gma.GMA_F32]) + _align((304 + BH) * K * 65 * 4)
        for dt in (gma.GMA_F32, gma.GMA_BF16):
            for op in (gma.OP_RESPONSIBILITIES, gma.OP_CAUSAL, gma.OP_CAUSAL_DECODE):
                assert on[op, dt] == off[op, dt], op
            for op in (gma.OP_BACKWARD_BIDIR, gma.OP_BACKWARD_CAUSAL, gma.OP_PROJECTED_BIDIR):
                assert on[op, dt] > off[op, dt], op
        # the key length does not enter the deterministic workspace either
        assert gma.workspace_bytes(P(N=1 << 20), gma.OP_BIDIR) == gma.workspace_bytes(P(N=128), gma.OP_BIDIR)
        for bad in (2, -2, 100):
            assert L.gma_set_deterministic(bad) == gma.GMA_ERR_INVALID_ARG
        assert L.gma_get_deterministic() == 1
        with pytest.raises(gma.GmaError):
            gma.set_deterministic(5)
    finally:
        assert L.gma_set_deterministic(-1) == gma.GMA_OK
    assert L.gma_get_deterministic() == default


def test_deterministic_environment_variable():
    """GMA_DETERMINISTIC sets the default of a fresh process: anything but "" or "0" turns it on."""
    code = ("from gaussian_mixture_sequence_gma_gb300 import gma; print(int(gma.deterministic()))")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for val, want in (("1", 1), ("yes", 1), ("0", 0), ("", 0)):
        env = dict(os.environ, GMA_DETERMINISTIC=val)
        out = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True,
                             timeout=120)
        assert out.returncode == 0, out.stderr
        assert int(out.stdout.strip().splitlines()[-1]) == want, val


def test_bounds_record_is_absent_from_the_normal_build(L):
    """The bounds-check entry points exist in every build and answer GMA_ERR_UNSUPPORTED in the normal one."""
    buf = (ctypes.c_ulonglong * 4)()
    assert L.gma_debug_bounds_read(buf) == gma.GMA_ERR_UNSUPPORTED
    assert L.gma_debug_bounds_clear() == gma.GMA_ERR_UNSUPPORTED
    assert L.gma_debug_bounds_selftest(None) == gma.GMA_ERR_UNSUPPORTED
    assert gma.bounds_record() is None
    assert gma.lib_path().endswith("libgma.so")
