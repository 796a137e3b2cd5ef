"""Thin Python binding over libgma.so (ctypes).

Argument marshalling only: PyTorch provides device memory, the current stream
and the workspace; every step of the GMA forward pass runs in the library's
CUDA kernels.  If ``libgma.so`` has not been built this module raises; there is
no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

# GMA_LIBRARY=checked loads the bounds-check debug build (libgma_checked.so) instead
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib",
                         "libgma_checked.so" if os.environ.get("GMA_LIBRARY") == "checked" else "libgma.so")

GMA_OK, GMA_ERR_INVALID_ARG, GMA_ERR_UNSUPPORTED, GMA_ERR_WORKSPACE, GMA_ERR_CUDA, GMA_ERR_TIMEOUT, GMA_ERR_RANGE = range(7)
GMA_F32, GMA_BF16 = 0, 1
(OP_RESPONSIBILITIES, OP_BIDIR, OP_CAUSAL, OP_CROSS, OP_CAUSAL_STATE, OP_CAUSAL_DECODE, OP_BACKWARD_BIDIR,
 OP_BACKWARD_CAUSAL, OP_PROJECTED_BIDIR, OP_PROJECTED_CAUSAL) = range(10)

EXPORTED = ("gma_workspace_bytes", "gma_responsibilities", "gma_forward_bidir", "gma_forward_causal", "gma_forward_cross", "gma_state_bytes", "gma_causal_state", "gma_causal_decode", "gma_decode_prepare", "gma_causal_decode_prepared", "gma_backward_bidir", "gma_backward_causal",
            "gma_forward_projected",
            "gma_check_device_error", "gma_status_string", "gma_version", "gma_last_error", "gma_launch_count", "gma_profile_enable",
            "gma_profile_read", "gma_forward_bidir_static_ws", "gma_static_ws_capacity", "gma_static_ws_check_error",
            "gma_debug_withhold_first_load", "gma_probe_ex2_rate", "gma_set_wait_limit_ns", "gma_get_wait_limit_ns",
            "gma_set_deterministic", "gma_get_deterministic",
            "gma_debug_bounds_read", "gma_debug_bounds_clear", "gma_debug_bounds_selftest")


class GmaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == GMA_ERR_CUDA:
            try:
                detail = " [%s]" % lib().gma_last_error().decode()
            except Exception:  # pragma: no cover
                pass
        super().__init__("%s failed: %s (status %d)%s" % (where, status_string(status), status, detail))


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int), ("d", ctypes.c_int),
                ("dv", ctypes.c_int), ("K", ctypes.c_int), ("dtype", ctypes.c_int), ("eps", ctypes.c_float)]


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError("libgma.so is not built (expected at %s); run "
                           "gaussian_mixture_sequence_gma_gb300.build.build()" % _LIB_PATH)
    L = ctypes.CDLL(_LIB_PATH)
    vp, fp, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t
    pp = ctypes.POINTER(Problem)
    L.gma_workspace_bytes.argtypes = [pp, ctypes.c_int]
    L.gma_workspace_bytes.restype = sz
    L.gma_responsibilities.argtypes = [pp, vp, fp, fp, fp, fp, vp, sz, vp]
    L.gma_responsibilities.restype = ctypes.c_int
    for name in ("gma_forward_bidir", "gma_forward_causal"):
        f = getattr(L, name)
        f.argtypes = [pp, vp, vp, vp, fp, fp, fp, vp, vp, sz, vp]
        f.restype = ctypes.c_int
    L.gma_forward_cross.argtypes = [pp, ctypes.c_int, vp, vp, vp, fp, fp, fp, vp, vp, sz, vp]
    L.gma_forward_cross.restype = ctypes.c_int
    L.gma_state_bytes.argtypes = [pp]
    L.gma_state_bytes.restype = sz
    L.gma_causal_state.argtypes = [pp, vp, vp, fp, fp, fp, vp, vp, sz, vp]
    L.gma_causal_state.restype = ctypes.c_int
    L.gma_causal_decode.argtypes = [pp, vp, vp, vp, fp, fp, fp, vp, vp, vp, sz, vp]
    L.gma_causal_decode.restype = ctypes.c_int
    L.gma_decode_prepare.argtypes = [pp, fp, fp, fp, vp, sz, vp]
    L.gma_decode_prepare.restype = ctypes.c_int
    L.gma_causal_decode_prepared.argtypes = [pp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.gma_causal_decode_prepared.restype = ctypes.c_int
    L.gma_backward_bidir.argtypes = [pp, vp, vp, vp, fp, fp, fp, vp, vp, vp, vp, fp, fp, fp, vp, sz, vp]
    L.gma_backward_bidir.restype = ctypes.c_int
    L.gma_backward_causal.argtypes = L.gma_backward_bidir.argtypes
    L.gma_backward_causal.restype = ctypes.c_int
    L.gma_forward_projected.argtypes = [pp, ctypes.c_int, ctypes.c_int, vp, vp, fp, fp, fp, fp, vp, vp, sz, vp]
    L.gma_forward_projected.restype = ctypes.c_int
    L.gma_check_device_error.argtypes = [vp, vp]
    L.gma_check_device_error.restype = ctypes.c_int
    L.gma_status_string.argtypes = [ctypes.c_int]
    L.gma_status_string.restype = ctypes.c_char_p
    L.gma_last_error.argtypes = []
    L.gma_last_error.restype = ctypes.c_char_p
    L.gma_version.argtypes = []
    L.gma_version.restype = ctypes.c_int
    L.gma_forward_bidir_static_ws.argtypes = [pp, vp, vp, vp, fp, fp, fp, vp, vp]
    L.gma_forward_bidir_static_ws.restype = ctypes.c_int
    L.gma_static_ws_capacity.argtypes = []
    L.gma_static_ws_capacity.restype = sz
    L.gma_static_ws_check_error.argtypes = [vp]
    L.gma_static_ws_check_error.restype = ctypes.c_int
    L.gma_probe_ex2_rate.argtypes = [vp, ctypes.POINTER(ctypes.c_double)]
    L.gma_probe_ex2_rate.restype = ctypes.c_int
    L.gma_debug_withhold_first_load.argtypes = []
    L.gma_debug_withhold_first_load.restype = None
    L.gma_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.gma_set_wait_limit_ns.restype = ctypes.c_int
    L.gma_get_wait_limit_ns.argtypes = []
    L.gma_get_wait_limit_ns.restype = ctypes.c_uint64
    L.gma_debug_bounds_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
    L.gma_debug_bounds_read.restype = ctypes.c_int
    L.gma_debug_bounds_clear.argtypes = []
    L.gma_debug_bounds_clear.restype = ctypes.c_int
    L.gma_debug_bounds_selftest.argtypes = [ctypes.c_void_p]
    L.gma_debug_bounds_selftest.restype = ctypes.c_int
    L.gma_set_deterministic.argtypes = [ctypes.c_int]
    L.gma_set_deterministic.restype = ctypes.c_int
    L.gma_get_deterministic.argtypes = []
    L.gma_get_deterministic.restype = ctypes.c_int
    L.gma_launch_count.argtypes = []
    L.gma_launch_count.restype = ctypes.c_ulonglong
    L.gma_profile_enable.argtypes = [ctypes.c_int]
    L.gma_profile_enable.restype = ctypes.c_int
    L.gma_profile_read.argtypes = [ctypes.c_char_p, ctypes.c_size_t]
    L.gma_profile_read.restype = ctypes.c_int
    _lib = L
    return L


def status_string(s: int) -> str:
    try:
        return lib().gma_status_string(int(s)).decode()
    except RuntimeError:
        return "status %d" % s


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return GMA_F32
    if t == torch.bfloat16:
        return GMA_BF16
    raise TypeError("GMA I/O dtype must be float32 or bfloat16, got %s" % t)


def problem(B, H, N, K, dtype, eps=1e-6, d=64, dv=64) -> Problem:
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return Problem(int(B), int(H), int(N), int(d), int(dv), int(K), int(code), float(eps))


def workspace_bytes(prob: Problem, op: int) -> int:
    return int(lib().gma_workspace_bytes(ctypes.byref(prob), int(op)))


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check_cuda(*ts):
    dev = None
    for t in ts:
        if not t.is_cuda:
            raise ValueError("GMA tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("GMA tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("GMA tensors must share one device")
    return dev


def _stream_handle(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def alloc_workspace(prob: Problem, op: int, device) -> torch.Tensor:
    n = workspace_bytes(prob, op)
    if n == 0:
        raise GmaError(GMA_ERR_INVALID_ARG, "gma_workspace_bytes")
    # torch's caching allocator returns 512-byte aligned blocks, above the 256 the ABI needs
    return torch.empty(n, dtype=torch.uint8, device=device)


def _params(mu, sigma2, log_pi):
    for t in (mu, sigma2, log_pi):
        if t.dtype != torch.float32:
            raise TypeError("mu, sigma2 and log_pi must be float32")
    return mu, sigma2, log_pi


def responsibilities(X, mu, sigma2, log_pi, out=None, workspace=None, stream=None):
    """Gamma [B,H,N,K] float32 of routing vectors X [B,H,N,64] (float32 or bf16)."""
    B, H, N, d = X.shape
    K = mu.shape[1]
    _params(mu, sigma2, log_pi)
    dev = _check_cuda(X, mu, sigma2, log_pi)
    prob = problem(B, H, N, K, X.dtype, 0.0, d=d)
    if out is None:
        out = torch.empty((B, H, N, K), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(prob, OP_RESPONSIBILITIES, dev)
    with torch.cuda.device(dev):
        s = lib().gma_responsibilities(ctypes.byref(prob), _ptr(X), _ptr(mu), _ptr(sigma2), _ptr(log_pi), _ptr(out),
                                       _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, "gma_responsibilities")
    return out


def _forward(name, op, Q, K, V, mu, sigma2, log_pi, eps, out, workspace, stream):
    B, H, N, d = Q.shape
    dv = V.shape[-1]
    Kc = mu.shape[1]
    _params(mu, sigma2, log_pi)
    dev = _check_cuda(Q, K, V, mu, sigma2, log_pi)
    if K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise TypeError("Q, K and V must share one dtype")
    prob = problem(B, H, N, Kc, Q.dtype, eps, d=d, dv=dv)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=Q.dtype, device=dev)
    if workspace is None:
        workspace = alloc_workspace(prob, op, dev)
    with torch.cuda.device(dev):
        s = getattr(lib(), name)(ctypes.byref(prob), _ptr(Q), _ptr(K), _ptr(V), _ptr(mu), _ptr(sigma2), _ptr(log_pi),
                                 _ptr(out), _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, name)
    return out


def forward_bidir(Q, K, V, mu, sigma2, log_pi, eps=1e-6, out=None, workspace=None, stream=None):
    """Bidirectional GMA forward: O [B,H,N,64] in the dtype of Q."""
    return _forward("gma_forward_bidir", OP_BIDIR, Q, K, V, mu, sigma2, log_pi, eps, out, workspace, stream)


def forward_causal(Q, K, V, mu, sigma2, log_pi, eps=1e-6, out=None, workspace=None, stream=None):
    """Causal GMA forward (inclusive prefix over key positions): O [B,H,N,64]."""
    return _forward("gma_forward_causal", OP_CAUSAL, Q, K, V, mu, sigma2, log_pi, eps, out, workspace, stream)


def forward_cross(Q, K, V, mu, sigma2, log_pi, eps=1e-6, out=None, workspace=None, stream=None):
    """Cross-attention GMA forward: queries Q [B,H,N,64] read the memory written by K [B,H,Nk,64] and
    V [B,H,Nk,64]; O [B,H,N,64] in the dtype of Q."""
    B, H, N, d = Q.shape
    Nk = K.shape[2]
    dv = V.shape[-1]
    Kc = mu.shape[1]
    _params(mu, sigma2, log_pi)
    dev = _check_cuda(Q, K, V, mu, sigma2, log_pi)
    if K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise TypeError("Q, K and V must share one dtype")
    if tuple(K.shape[:2]) != (B, H) or tuple(V.shape[:3]) != (B, H, Nk):
        raise ValueError("K [B,H,Nk,d] and V [B,H,Nk,dv] must match Q's batch and heads")
    prob = problem(B, H, N, Kc, Q.dtype, eps, d=d, dv=dv)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=Q.dtype, device=dev)
    if workspace is None:
        workspace = alloc_workspace(prob, OP_CROSS, dev)
    with torch.cuda.device(dev):
        s = lib().gma_forward_cross(ctypes.byref(prob), int(Nk), _ptr(Q), _ptr(K), _ptr(V), _ptr(mu), _ptr(sigma2),
                                    _ptr(log_pi), _ptr(out), _ptr(workspace), workspace.numel(),
                                    _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, "gma_forward_cross")
    return out


def forward_projected(X, Wqkv, bqkv, mu, sigma2, log_pi, causal, eps=1e-6, out=None, workspace=None, stream=None):
    """Transformer-block form: Q, K, V = split_heads(X Wqkv + bqkv) then the GMA forward.  X [B,N,dm] and
    Wqkv [dm, 3*H*64] in the I/O dtype (column blocks Q | K | V, head h = columns 64h..64h+63 of a
    block), bqkv [3*H*64] float32; O [B,H,N,64] in the I/O dtype."""
    B, N, dm = X.shape
    Kc = mu.shape[1]
    H = mu.shape[0]
    _params(mu, sigma2, log_pi)
    dev = _check_cuda(X, Wqkv, bqkv, mu, sigma2, log_pi)
    if Wqkv.dtype != X.dtype or bqkv.dtype != torch.float32:
        raise TypeError("Wqkv must have X's dtype and bqkv must be float32")
    if tuple(Wqkv.shape) != (dm, 3 * H * 64) or tuple(bqkv.shape) != (3 * H * 64,):
        raise ValueError("Wqkv must be [dm, 3*H*64] and bqkv [3*H*64] (H from mu)")
    prob = problem(B, H, N, Kc, X.dtype, eps)
    op = OP_PROJECTED_CAUSAL if causal else OP_PROJECTED_BIDIR
    if out is None:
        out = torch.empty((B, H, N, 64), dtype=X.dtype, device=dev)
    if workspace is None:
        workspace = alloc_workspace(prob, op, dev)
    with torch.cuda.device(dev):
        s = lib().gma_forward_projected(ctypes.byref(prob), 1 if causal else 0, int(dm), _ptr(X), _ptr(Wqkv),
                                        _ptr(bqkv), _ptr(mu), _ptr(sigma2), _ptr(log_pi), _ptr(out),
                                        _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, "gma_forward_projected")
    return out


def causal_state(K, V, mu, sigma2, log_pi, state=None, workspace=None, stream=None):
    """State float32 [B,H,Kc,65] (latent memory | normaliser) after the N keys / values of K, V [B,H,N,64]."""
    B, H, N, d = K.shape
    dv = V.shape[-1]
    Kc = mu.shape[1]
    _params(mu, sigma2, log_pi)
    dev = _check_cuda(K, V, mu, sigma2, log_pi)
    if V.dtype != K.dtype:
        raise TypeError("K and V must share one dtype")
    prob = problem(B, H, N, Kc, K.dtype, 0.0, d=d, dv=dv)
    if state is None:
        state = torch.empty((B, H, Kc, dv + 1), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(prob, OP_CAUSAL_STATE, dev)
    with torch.cuda.device(dev):
        s = lib().gma_causal_state(ctypes.byref(prob), _ptr(K), _ptr(V), _ptr(mu), _ptr(sigma2), _ptr(log_pi),
                                   _ptr(state), _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, "gma_causal_state")
    return state


def causal_decode(Q, K, V, mu, sigma2, log_pi, state, eps=1e-6, out=None, workspace=None, stream=None):
    """Decode the N new tokens of Q, K, V [B,H,N,64] in order against `state` (float32 [B,H,Kc,65],
    updated in place); returns O [B,H,N,64], each row the causal output of its position."""
    B, H, N, d = Q.shape
    dv = V.shape[-1]
    Kc = mu.shape[1]
    _params(mu, sigma2, log_pi)
    dev = _check_cuda(Q, K, V, mu, sigma2, log_pi, state)
    if K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise TypeError("Q, K and V must share one dtype")
    if state.dtype != torch.float32 or tuple(state.shape) != (B, H, Kc, dv + 1):
        raise ValueError("state must be float32 [B,H,K,dv+1]")
    prob = problem(B, H, N, Kc, Q.dtype, eps, d=d, dv=dv)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=Q.dtype, device=dev)
    if workspace is None:
        workspace = alloc_workspace(prob, OP_CAUSAL_DECODE, dev)
    with torch.cuda.device(dev):
        s = lib().gma_causal_decode(ctypes.byref(prob), _ptr(Q), _ptr(K), _ptr(V), _ptr(mu), _ptr(sigma2),
                                    _ptr(log_pi), _ptr(state), _ptr(out), _ptr(workspace), workspace.numel(),
                                    _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, "gma_causal_decode")
    return out


def decode_prepare(mu, sigma2, log_pi, dtype=torch.bfloat16, workspace=None, stream=None):
    """Fold the parameters once for causal_decode_prepared; returns the decode workspace holding them
    (valid for any B and dtype with these H and K, as long as the parameters do not change)."""
    H, Kc, d = mu.shape
    _params(mu, sigma2, log_pi)
    dev = _check_cuda(mu, sigma2, log_pi)
    prob = problem(1, H, 1, Kc, dtype, 1e-6, d=d, dv=d)
    if workspace is None:
        workspace = alloc_workspace(prob, OP_CAUSAL_DECODE, dev)
    with torch.cuda.device(dev):
        s = lib().gma_decode_prepare(ctypes.byref(prob), _ptr(mu), _ptr(sigma2), _ptr(log_pi), _ptr(workspace),
                                     workspace.numel(), _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, "gma_decode_prepare")
    return workspace


def causal_decode_prepared(Q, K, V, state, workspace, eps=1e-6, out=None, stream=None):
    """causal_decode with the parameters folded by decode_prepare into `workspace` (one launch)."""
    B, H, N, d = Q.shape
    dv = V.shape[-1]
    Kc = state.shape[2]
    dev = _check_cuda(Q, K, V, state, workspace)
    if K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise TypeError("Q, K and V must share one dtype")
    if state.dtype != torch.float32 or tuple(state.shape) != (B, H, Kc, dv + 1):
        raise ValueError("state must be float32 [B,H,K,dv+1]")
    prob = problem(B, H, N, Kc, Q.dtype, eps, d=d, dv=dv)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=Q.dtype, device=dev)
    with torch.cuda.device(dev):
        s = lib().gma_causal_decode_prepared(ctypes.byref(prob), _ptr(Q), _ptr(K), _ptr(V), _ptr(state), _ptr(out),
                                             _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, "gma_causal_decode_prepared")
    return out


def backward_causal(Q, K, V, mu, sigma2, log_pi, dO, eps=1e-6, workspace=None, stream=None):
    """Gradients (dQ, dK, dV, dmu, dsigma2, dlog_pi) of the causal forward given dO [B,H,N,64]."""
    return backward_bidir(Q, K, V, mu, sigma2, log_pi, dO, eps, workspace, stream, causal=True)


def backward_bidir(Q, K, V, mu, sigma2, log_pi, dO, eps=1e-6, workspace=None, stream=None, causal=False):
    """Gradients (dQ, dK, dV, dmu, dsigma2, dlog_pi) of the bidirectional forward given dO [B,H,N,64]."""
    B, H, N, d = Q.shape
    dv = V.shape[-1]
    Kc = mu.shape[1]
    _params(mu, sigma2, log_pi)
    dev = _check_cuda(Q, K, V, mu, sigma2, log_pi, dO)
    if K.dtype != Q.dtype or V.dtype != Q.dtype or dO.dtype != Q.dtype:
        raise TypeError("Q, K, V and dO must share one dtype")
    prob = problem(B, H, N, Kc, Q.dtype, eps, d=d, dv=dv)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    dmu, dsigma2, dlog_pi = torch.empty_like(mu), torch.empty_like(sigma2), torch.empty_like(log_pi)
    name = "gma_backward_causal" if causal else "gma_backward_bidir"
    if workspace is None:
        workspace = alloc_workspace(prob, OP_BACKWARD_CAUSAL if causal else OP_BACKWARD_BIDIR, dev)
    with torch.cuda.device(dev):
        s = getattr(lib(), name)(ctypes.byref(prob), _ptr(Q), _ptr(K), _ptr(V), _ptr(mu), _ptr(sigma2),
                                     _ptr(log_pi), _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dmu), _ptr(dsigma2),
                                     _ptr(dlog_pi), _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, name)
    return dQ, dK, dV, dmu, dsigma2, dlog_pi


def forward_bidir_static_ws(Q, K, V, mu, sigma2, log_pi, eps=1e-6, out=None, stream=None):
    """Bidirectional forward whose scratch is the library's own static device array (no workspace
    is allocated anywhere); see gma_forward_bidir_static_ws in gma.h for its limits."""
    B, H, N, d = Q.shape
    dv = V.shape[-1]
    _params(mu, sigma2, log_pi)
    # the library reads K and V with Q's element size; a mismatch would read past their buffers
    if K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise TypeError("Q, K and V must share one dtype")
    if tuple(K.shape) != (B, H, N, d) or tuple(V.shape[:3]) != (B, H, N):
        raise ValueError("K must be [B,H,N,d] and V [B,H,N,dv] with Q's B, H, N")
    if out is not None and (out.dtype != Q.dtype or tuple(out.shape) != (B, H, N, dv)):
        raise TypeError("out must have Q's dtype and shape [B,H,N,dv]")
    dev = _check_cuda(Q, K, V, mu, sigma2, log_pi) if out is None else _check_cuda(Q, K, V, mu, sigma2, log_pi, out)
    prob = problem(B, H, N, mu.shape[1], Q.dtype, eps, d=d, dv=dv)
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=Q.dtype, device=dev)
    with torch.cuda.device(dev):
        s = lib().gma_forward_bidir_static_ws(ctypes.byref(prob), _ptr(Q), _ptr(K), _ptr(V), _ptr(mu), _ptr(sigma2),
                                              _ptr(log_pi), _ptr(out), _stream_handle(stream, dev))
    if s != GMA_OK:
        raise GmaError(s, "gma_forward_bidir_static_ws")
    return out


def static_ws_capacity() -> int:
    return int(lib().gma_static_ws_capacity())


def static_ws_check_error(stream=None, device=None) -> int:
    """Synchronises the stream and returns the status held in the library-held array's error word
    (the array used by forward_bidir_static_ws on the current device)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().gma_static_ws_check_error(_stream_handle(stream, dev)))


def check_device_error(workspace, stream=None) -> int:
    """Synchronises the stream and returns the status held in the workspace's error word."""
    dev = workspace.device
    with torch.cuda.device(dev):
        return int(lib().gma_check_device_error(_ptr(workspace), _stream_handle(stream, dev)))


def set_wait_limit_ns(ns: int) -> None:
    """Process-wide limit of the bf16 kernels' bounded device waits (0: the default, GMA_WAIT_LIMIT_MS or 1 s)."""
    st = int(lib().gma_set_wait_limit_ns(int(ns)))
    if st != GMA_OK:
        raise GmaError(st, "gma_set_wait_limit_ns")


def wait_limit_ns() -> int:
    return int(lib().gma_get_wait_limit_ns())


def bounds_record() -> tuple[int, int, int, int] | None:
    """Bounds-check debug build: (first failing site, its index, its extent, failures); None in the
    normal build."""
    out = (ctypes.c_ulonglong * 4)()
    st = int(lib().gma_debug_bounds_read(out))
    if st == GMA_ERR_UNSUPPORTED:
        return None
    if st != GMA_OK:
        raise GmaError(st, "gma_debug_bounds_read")
    return tuple(int(v) for v in out)


def set_deterministic(mode: int) -> None:
    """Process-wide deterministic reduction mode: 1 on, 0 off, -1 the default (GMA_DETERMINISTIC).

    With it on, sums across CTAs are taken in a fixed order and repeated calls give bitwise-equal
    outputs; workspaces grow, so a workspace sized before the switch may be too small."""
    st = int(lib().gma_set_deterministic(int(mode)))
    if st != GMA_OK:
        raise GmaError(st, "gma_set_deterministic")


def deterministic() -> bool:
    return bool(lib().gma_get_deterministic())


def launch_count() -> int:
    """Kernels launched by libgma.so so far in this process."""
    return int(lib().gma_launch_count())


def profile_enable(on: bool) -> None:
    s = lib().gma_profile_enable(1 if on else 0)
    if s != GMA_OK:
        raise GmaError(s, "gma_profile_enable")


def profile_read() -> dict:
    """{kernel name: (launches, total ms)} of the launches recorded while profiling was on."""
    buf = ctypes.create_string_buffer(1 << 16)
    n = lib().gma_profile_read(buf, len(buf))
    if n < 0:
        raise GmaError(GMA_ERR_CUDA, "gma_profile_read")
    out = {}
    for line in buf.value.decode().splitlines():
        name, cnt, ms = line.split()
        out[name] = (int(cnt), float(ms))
    return out


def probe_ex2_rate(device=None) -> float:
    """Exponentials per second of the GPU's ex2 unit (all SMs), measured now."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    out = ctypes.c_double(0.0)
    with torch.cuda.device(dev):
        s = lib().gma_probe_ex2_rate(_stream_handle(None, dev), ctypes.byref(out))
    if s != GMA_OK:
        raise GmaError(s, "gma_probe_ex2_rate")
    return float(out.value)
