"""Thin ctypes binding of libm2rnn.so (include/m2rnn.h).

The ``m2rnn_*`` functions mirror the C ABI one to one (raw device pointers and
sizes).  ``forward`` / ``backward`` are torch conveniences on top: they take
contiguous CUDA tensors, allocate outputs and the workspace with torch (device
memory and streams are all torch is used for) and call the C ABI on the
current stream.  Every step of both scans runs in the library's CUDA kernels;
there is no CPU path.  Loading fails loudly when the library is missing.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libm2rnn.so")

M2RNN_OK = 0
M2RNN_ERR_INVALID_ARG = -1
M2RNN_ERR_UNSUPPORTED = -2
M2RNN_ERR_WORKSPACE = -3
M2RNN_ERR_CUDA = -4
M2RNN_ERR_TIMEOUT = -5
M2RNN_ERR_DEVICE = -6
M2RNN_F32 = 0
M2RNN_BF16 = 1
M2RNN_OPT_KERNEL_FAMILY = 0
M2RNN_OPT_TEST_STALL_TILE = 1
# Kernel family codes (as m2rnn_path returns them); -1 = automatic choice.
FAMILIES = {"auto": -1, "simt": 0, "tcgen05": 1, "mma": 2}

EXPORTS = (
    "m2rnn_version", "m2rnn_status_string", "m2rnn_checkpoint_count", "m2rnn_path",
    "m2rnn_forward_workspace_size", "m2rnn_backward_workspace_size", "m2rnn_forward",
    "m2rnn_backward", "m2rnn_sync_status", "m2rnn_forward_state", "m2rnn_backward_state",
    "m2rnn_decode_step", "m2rnn_backward_state_workspace_size", "m2rnn_forward_gated",
    "m2rnn_backward_gated", "m2rnn_output_norm", "m2rnn_output_norm_backward_workspace_size",
    "m2rnn_output_norm_backward", "m2rnn_z_stash_size", "m2rnn_set_option",
    "m2rnn_backward_noalloc", "m2rnn_backward_noalloc_status",
)

_lib = None


class M2RNNError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Load libm2rnn.so (built in-tree); raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -m matrix_state_non_gb300.build` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, ci, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.m2rnn_version.restype = ci
    lib.m2rnn_version.argtypes = []
    lib.m2rnn_status_string.restype = ctypes.c_char_p
    lib.m2rnn_status_string.argtypes = [ci]
    lib.m2rnn_checkpoint_count.restype = i64
    lib.m2rnn_checkpoint_count.argtypes = [i64, ci]
    lib.m2rnn_path.restype = ci
    lib.m2rnn_path.argtypes = [i64, i64, ci]
    lib.m2rnn_set_option.restype = ci
    lib.m2rnn_set_option.argtypes = [ci, ci, ctypes.POINTER(ci)]
    lib.m2rnn_forward_workspace_size.restype = sz
    lib.m2rnn_forward_workspace_size.argtypes = [i64, i64, i64, i64, i64, ci]
    lib.m2rnn_backward_workspace_size.restype = sz
    lib.m2rnn_backward_workspace_size.argtypes = [i64, i64, i64, i64, i64, ci, ci, ci]
    lib.m2rnn_forward.restype = ci
    lib.m2rnn_forward.argtypes = [vp] * 9 + [ci] + [i64] * 5 + [ci, vp, sz, vp]
    lib.m2rnn_backward.restype = ci
    lib.m2rnn_backward.argtypes = [vp] * 9 + [ci] + [vp] * 6 + [i64] * 5 + [ci, vp, sz, vp]
    lib.m2rnn_sync_status.restype = ci
    lib.m2rnn_sync_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.m2rnn_forward_state.restype = ci
    lib.m2rnn_forward_state.argtypes = [vp] * 10 + [ci, vp] + [i64] * 6 + [ci, vp, sz, vp]
    lib.m2rnn_backward_state.restype = ci
    lib.m2rnn_backward_state.argtypes = [vp] * 10 + [ci, vp] + [vp] * 7 + [ctypes.c_float] + [i64] * 6 + [ci, vp, sz, vp]
    lib.m2rnn_backward_state_workspace_size.restype = sz
    lib.m2rnn_backward_state_workspace_size.argtypes = [i64] * 6 + [ci, ci, ci]
    lib.m2rnn_decode_step.restype = ci
    lib.m2rnn_decode_step.argtypes = [vp] * 8 + [i64] * 5 + [ci, vp, sz, vp]
    fl = ctypes.c_float
    lib.m2rnn_forward_gated.restype = ci
    lib.m2rnn_forward_gated.argtypes = [vp] * 12 + [ci, vp] + [i64] * 6 + [ci, vp, sz, vp]
    lib.m2rnn_backward_gated.restype = ci
    lib.m2rnn_backward_gated.argtypes = [vp] * 12 + [ci, vp] + [vp] * 9 + [fl] + [i64] * 6 + [ci, vp, sz, vp]
    lib.m2rnn_z_stash_size.restype = sz
    lib.m2rnn_z_stash_size.argtypes = [i64] * 5 + [ci]
    lib.m2rnn_output_norm.restype = ci
    lib.m2rnn_output_norm.argtypes = [vp] * 3 + [fl] + [vp] * 2 + [i64] * 4 + [ci, vp]
    lib.m2rnn_output_norm_backward_workspace_size.restype = sz
    lib.m2rnn_output_norm_backward_workspace_size.argtypes = [i64] * 4
    lib.m2rnn_output_norm_backward.restype = ci
    lib.m2rnn_output_norm_backward.argtypes = [vp] * 4 + [fl] + [vp] * 3 + [i64] * 4 + [ci, vp, sz, vp]
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# One-to-one wrappers of the C ABI (integers are device addresses).
# ---------------------------------------------------------------------------
def m2rnn_version() -> int:
    return load().m2rnn_version()


def status_string(status: int) -> str:
    return load().m2rnn_status_string(status).decode()


m2rnn_status_string = status_string


def m2rnn_checkpoint_count(T: int, ckpt_every: int) -> int:
    return load().m2rnn_checkpoint_count(T, ckpt_every)


def m2rnn_path(K: int, V: int, dtype: int) -> int:
    return load().m2rnn_path(K, V, dtype)


def m2rnn_set_option(option: int, value: int):
    """Returns (status, previous value)."""
    prev = ctypes.c_int(0)
    st = load().m2rnn_set_option(option, value, ctypes.byref(prev))
    return st, prev.value


@contextlib.contextmanager
def kernel_family(name: str):
    """Run the enclosed calls on one kernel family ("auto", "tcgen05", "mma",
    "simt"); the previous choice is restored on exit."""
    st, prev = m2rnn_set_option(M2RNN_OPT_KERNEL_FAMILY, FAMILIES[name])
    _check(st, "m2rnn_set_option")
    try:
        yield
    finally:
        m2rnn_set_option(M2RNN_OPT_KERNEL_FAMILY, prev)


@contextlib.contextmanager
def stall_tile_hook(tile: int):
    """Failure-detection test hook (see include/m2rnn.h): the warp-MMA forward
    withholds input tile `tile` of single-CTA chains inside the block."""
    st, prev = m2rnn_set_option(M2RNN_OPT_TEST_STALL_TILE, tile)
    _check(st, "m2rnn_set_option")
    try:
        yield
    finally:
        m2rnn_set_option(M2RNN_OPT_TEST_STALL_TILE, prev)


def m2rnn_forward_workspace_size(B, T, N, K, V, dtype) -> int:
    return load().m2rnn_forward_workspace_size(B, T, N, K, V, dtype)


def m2rnn_backward_workspace_size(B, T, N, K, V, dtype, ckpt_every, have_ckpt) -> int:
    return load().m2rnn_backward_workspace_size(B, T, N, K, V, dtype, ckpt_every, int(bool(have_ckpt)))


def m2rnn_forward(q, k, v, f, W, w_r, y, H_T, ckpt, ckpt_every, B, T, N, K, V, dtype,
                  workspace, workspace_bytes, stream) -> int:
    return load().m2rnn_forward(q, k, v, f, W, w_r, y, H_T, ckpt, ckpt_every, B, T, N, K, V,
                                dtype, workspace, workspace_bytes, stream)


def m2rnn_backward(q, k, v, f, W, w_r, dy, dH_T, ckpt, ckpt_every, dq, dk, dv, df, dW, dw_r,
                   B, T, N, K, V, dtype, workspace, workspace_bytes, stream) -> int:
    return load().m2rnn_backward(q, k, v, f, W, w_r, dy, dH_T, ckpt, ckpt_every, dq, dk, dv,
                                 df, dW, dw_r, B, T, N, K, V, dtype, workspace,
                                 workspace_bytes, stream)


def m2rnn_forward_state(q, k, v, f, W, w_r, H_0, y, H_T, ckpt, ckpt_every, z_stash, B, T, N, qk_heads, K, V,
                        dtype, workspace, workspace_bytes, stream) -> int:
    return load().m2rnn_forward_state(q, k, v, f, W, w_r, H_0, y, H_T, ckpt, ckpt_every, z_stash, B, T, N,
                                      qk_heads, K, V, dtype, workspace, workspace_bytes, stream)


def m2rnn_z_stash_size(B, T, N, K, V, dtype) -> int:
    return load().m2rnn_z_stash_size(B, T, N, K, V, dtype)


def m2rnn_backward_state_workspace_size(B, T, N, qk_heads, K, V, dtype, ckpt_every, have_ckpt) -> int:
    return load().m2rnn_backward_state_workspace_size(B, T, N, qk_heads, K, V, dtype, ckpt_every,
                                                      int(bool(have_ckpt)))


def m2rnn_backward_state(q, k, v, f, W, w_r, H_0, dy, dH_T, ckpt, ckpt_every, z_stash, dq, dk, dv, df, dW,
                         dw_r, dH_0, state_grad_clip, B, T, N, qk_heads, K, V, dtype, workspace,
                         workspace_bytes, stream) -> int:
    return load().m2rnn_backward_state(q, k, v, f, W, w_r, H_0, dy, dH_T, ckpt, ckpt_every, z_stash, dq, dk,
                                       dv, df, dW, dw_r, dH_0, state_grad_clip, B, T, N, qk_heads, K,
                                       V, dtype, workspace, workspace_bytes, stream)


def m2rnn_decode_step(H, q, k, v, f, W, w_r, y, B, N, qk_heads, K, V, dtype, workspace,
                      workspace_bytes, stream) -> int:
    return load().m2rnn_decode_step(H, q, k, v, f, W, w_r, y, B, N, qk_heads, K, V, dtype, workspace,
                                    workspace_bytes, stream)


def m2rnn_forward_gated(q, k, v, a, alpha, beta, W, w_r, H_0, y, H_T, ckpt, ckpt_every, z_stash, B, T, N,
                        qk_heads, K, V, dtype, workspace, workspace_bytes, stream) -> int:
    return load().m2rnn_forward_gated(q, k, v, a, alpha, beta, W, w_r, H_0, y, H_T, ckpt, ckpt_every, z_stash, B, T,
                                      N, qk_heads, K, V, dtype, workspace, workspace_bytes, stream)


def m2rnn_backward_gated(q, k, v, a, alpha, beta, W, w_r, H_0, dy, dH_T, ckpt, ckpt_every, z_stash, dq, dk, dv,
                         da, dalpha, dbeta, dW, dw_r, dH_0, state_grad_clip, B, T, N, qk_heads, K, V, dtype,
                         workspace, workspace_bytes, stream) -> int:
    return load().m2rnn_backward_gated(q, k, v, a, alpha, beta, W, w_r, H_0, dy, dH_T, ckpt, ckpt_every, z_stash,
                                       dq, dk, dv, da, dalpha, dbeta, dW, dw_r, dH_0, state_grad_clip, B, T, N,
                                       qk_heads, K, V, dtype, workspace, workspace_bytes, stream)


def m2rnn_output_norm(y, g, w, eps, out, rstd, B, T, N, V, dtype, stream) -> int:
    return load().m2rnn_output_norm(y, g, w, eps, out, rstd, B, T, N, V, dtype, stream)


def m2rnn_output_norm_backward_workspace_size(B, T, N, V) -> int:
    return load().m2rnn_output_norm_backward_workspace_size(B, T, N, V)


def m2rnn_output_norm_backward(y, g, w, dout, eps, dy, dg, dw, B, T, N, V, dtype, workspace,
                               workspace_bytes, stream) -> int:
    return load().m2rnn_output_norm_backward(y, g, w, dout, eps, dy, dg, dw, B, T, N, V, dtype, workspace,
                                             workspace_bytes, stream)


def m2rnn_sync_status(workspace, stream):
    """Returns (status, detail)."""
    d = ctypes.c_uint32(0)
    st = load().m2rnn_sync_status(workspace, stream, ctypes.byref(d))
    return st, d.value


# ---------------------------------------------------------------------------
# torch conveniences
# ---------------------------------------------------------------------------
def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return M2RNN_BF16
    if t.dtype == torch.float32:
        return M2RNN_F32
    raise TypeError(f"unsupported input dtype {t.dtype}")


def _check(st: int, what: str):
    if st != M2RNN_OK:
        raise M2RNNError(st, what)


def _stream_handle(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _shapes(q, v):
    """(B, T, N, K, V, qk_heads): N from v; q, k carry 1 head when shared."""
    B, T, _, K = q.shape
    N, V = v.shape[2], v.shape[-1]
    return B, T, N, K, V, q.shape[2]


def forward(q, k, v, f, W, w_r, *, H_0=None, want_state: bool = True, ckpt_every: int = 0,
            gate=None, stash: bool = False, out=None, workspace=None, stream=None):
    """Forward scan on the GPU from ``H_0`` (fp32 [B,N,K,V]; None = zero).
    Returns dict(y, H_T[, ckpt]).

    ``ckpt_every`` > 0 also writes the checkpoints the backward can reuse.
    ``gate`` = (a, alpha, beta) with ``f`` None computes the forget gate in
    the kernels (m2rnn_forward_gated).  ``stash`` also returns "z_stash", the
    fp16 Z_t of every step for ``backward`` (bf16, V = 64 only).  ``out`` may
    hold preallocated y / H_T / ckpt / z_stash tensors.
    """
    import torch
    B, T, N, K, V, NQ = _shapes(q, v)
    dt = _dtype_code(q)
    dev = q.device
    out = dict(out or {})
    y = out.get("y")
    if y is None:
        y = torch.empty((B, T, N, V), device=dev, dtype=torch.float32)
    H_T = out.get("H_T")
    if H_T is None and want_state:
        H_T = torch.empty((B, N, K, V), device=dev, dtype=torch.float32)
    ckpt = out.get("ckpt")
    if ckpt is None and ckpt_every > 0:
        nck = m2rnn_checkpoint_count(T, ckpt_every)
        ckpt = torch.empty((B, N, max(nck, 0), K, V), device=dev, dtype=torch.float32)
    ws_bytes = m2rnn_forward_workspace_size(B, T, N, K, V, dt)
    if ws_bytes == 0:
        raise M2RNNError(M2RNN_ERR_INVALID_ARG, "m2rnn_forward_workspace_size")
    if workspace is None:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    z_stash = out.get("z_stash")
    if z_stash is None and stash:
        zb = m2rnn_z_stash_size(B, T, N, K, V, dt)
        if zb == 0:
            raise M2RNNError(M2RNN_ERR_UNSUPPORTED, "m2rnn_z_stash_size")
        z_stash = torch.empty(zb, device=dev, dtype=torch.uint8)
    ce = ckpt_every if ckpt is not None else 0
    if gate is not None:
        if f is not None:
            raise ValueError("give either f or gate=(a, alpha, beta), not both")
        a, alpha, beta = gate
        st = m2rnn_forward_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(alpha), _ptr(beta), _ptr(W),
                                 _ptr(w_r), _ptr(H_0), _ptr(y), _ptr(H_T), _ptr(ckpt), ce, _ptr(z_stash), B, T,
                                 N, NQ, K, V, dt, _ptr(workspace), workspace.numel(), _stream_handle(stream))
        _check(st, "m2rnn_forward_gated")
    else:
        st = m2rnn_forward_state(_ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(W), _ptr(w_r), _ptr(H_0),
                                 _ptr(y), _ptr(H_T), _ptr(ckpt), ce, _ptr(z_stash), B, T, N, NQ, K, V, dt,
                                 _ptr(workspace), workspace.numel(), _stream_handle(stream))
        _check(st, "m2rnn_forward_state")
    res = dict(y=y, H_T=H_T, workspace=workspace)
    if ckpt is not None:
        res["ckpt"] = ckpt
    if z_stash is not None:
        res["z_stash"] = z_stash
    return res


def backward(q, k, v, f, W, w_r, dy, *, dH_T=None, H_0=None, want_dH0: bool = False, ckpt=None,
             ckpt_every: int = 14, state_grad_clip: float = 0.0, gate=None, z_stash=None, out=None,
             workspace=None, stream=None):
    """Backward scan on the GPU.  Returns dict(dq, dk, dv, df, dW, dw_r[, dH_0]);
    with ``gate`` = (a, alpha, beta) (and ``f`` None) da, dalpha, dbeta
    replace df.

    ``H_0`` is the forward's initial state (None = zero); ``ckpt``, if given,
    must come from a forward with the same ``H_0`` (and gate); ``z_stash``, with
    that forward's ``ckpt``, replaces the rerun of the transform and tanh;
    ``state_grad_clip`` > 0 clamps every new state gradient C_{t-1} to [-c, c]."""
    import torch
    B, T, N, K, V, NQ = _shapes(q, v)
    dt = _dtype_code(q)
    dev = q.device
    out = dict(out or {})

    def _get(name, shape):
        t = out.get(name)
        return t if t is not None else torch.empty(shape, device=dev, dtype=torch.float32)

    dq = _get("dq", (B, T, NQ, K))
    dk = _get("dk", (B, T, NQ, K))
    dv = _get("dv", (B, T, N, V))
    df = _get("df", (B, T, N)) if gate is None else None
    dW = _get("dW", (N, V, V))
    dw_r = _get("dw_r", (N, V))
    dH_0 = _get("dH_0", (B, N, K, V)) if want_dH0 else None
    ws_bytes = m2rnn_backward_state_workspace_size(B, T, N, NQ, K, V, dt, ckpt_every, ckpt is not None)
    if ws_bytes == 0:
        raise M2RNNError(M2RNN_ERR_INVALID_ARG, "m2rnn_backward_state_workspace_size")
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    if gate is not None:
        if f is not None:
            raise ValueError("give either f or gate=(a, alpha, beta), not both")
        a, alpha, beta = gate
        da = _get("da", (B, T, N))
        dalpha = _get("dalpha", (N,))
        dbeta = _get("dbeta", (N,))
        st = m2rnn_backward_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(alpha), _ptr(beta), _ptr(W),
                                  _ptr(w_r), _ptr(H_0), _ptr(dy), _ptr(dH_T), _ptr(ckpt), ckpt_every,
                                  _ptr(z_stash), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(da), _ptr(dalpha), _ptr(dbeta), _ptr(dW),
                                  _ptr(dw_r), _ptr(dH_0), float(state_grad_clip), B, T, N, NQ, K, V, dt,
                                  _ptr(workspace), workspace.numel(), _stream_handle(stream))
        _check(st, "m2rnn_backward_gated")
        res = dict(dq=dq, dk=dk, dv=dv, da=da, dalpha=dalpha, dbeta=dbeta, dW=dW, dw_r=dw_r,
                   workspace=workspace)
    else:
        st = m2rnn_backward_state(_ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(W), _ptr(w_r), _ptr(H_0),
                                  _ptr(dy), _ptr(dH_T), _ptr(ckpt), ckpt_every, _ptr(z_stash), _ptr(dq),
                                  _ptr(dk), _ptr(dv), _ptr(df), _ptr(dW), _ptr(dw_r), _ptr(dH_0),
                                  float(state_grad_clip), B, T, N, NQ, K, V, dt, _ptr(workspace),
                                  workspace.numel(), _stream_handle(stream))
        _check(st, "m2rnn_backward_state")
        res = dict(dq=dq, dk=dk, dv=dv, df=df, dW=dW, dw_r=dw_r, workspace=workspace)
    if dH_0 is not None:
        res["dH_0"] = dH_0
    return res


def decode_step(H, q, k, v, f, W, w_r, *, y=None, workspace=None, stream=None):
    """One decoding step on the GPU: ``H`` (fp32 [B,N,K,V], contiguous) is
    updated in place; q, k [B,N,K] (or [B,1,K], shared by the heads),
    v [B,N,V], f [B,N].  Returns y [B,N,V]."""
    import torch
    B, NQ, K = q.shape
    N, V = v.shape[1], v.shape[-1]
    dt = _dtype_code(q)
    if y is None:
        y = torch.empty((B, N, V), device=q.device, dtype=torch.float32)
    ws_bytes = m2rnn_forward_workspace_size(B, 1, N, K, V, dt)
    if ws_bytes == 0:
        raise M2RNNError(M2RNN_ERR_INVALID_ARG, "m2rnn_forward_workspace_size")
    if workspace is None:
        workspace = torch.empty(ws_bytes, device=q.device, dtype=torch.uint8)
    st = m2rnn_decode_step(_ptr(H), _ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(W), _ptr(w_r), _ptr(y),
                           B, N, NQ, K, V, dt, _ptr(workspace), workspace.numel(),
                           _stream_handle(stream))
    _check(st, "m2rnn_decode_step")
    return y


def output_norm(y, g, w, *, eps: float = 1e-6, want_rstd: bool = False, out=None, stream=None):
    """out = w * (y*g) * rms^-1 over each token's N*V elements; y fp32
    [B,T,N,V], g [B,T,N,V] (bf16 or fp32), w fp32 [N,V].  Returns out, or
    (out, rstd [B,T]) with ``want_rstd``."""
    import torch
    B, T, N, V = y.shape
    if out is None:
        out = torch.empty((B, T, N, V), device=y.device, dtype=torch.float32)
    rstd = torch.empty((B, T), device=y.device, dtype=torch.float32) if want_rstd else None
    st = m2rnn_output_norm(_ptr(y), _ptr(g), _ptr(w), float(eps), _ptr(out), _ptr(rstd), B, T, N, V,
                           _dtype_code(g), _stream_handle(stream))
    _check(st, "m2rnn_output_norm")
    return (out, rstd) if want_rstd else out


def output_norm_backward(y, g, w, dout, *, eps: float = 1e-6, out=None, workspace=None, stream=None):
    """Returns dict(dy, dg [B,T,N,V], dw [N,V]) of ``output_norm``; ``out``
    may hold preallocated dy / dg / dw."""
    import torch
    B, T, N, V = y.shape
    dev = y.device
    out = dict(out or {})

    def _get(name, shape):
        t = out.get(name)
        return t if t is not None else torch.empty(shape, device=dev, dtype=torch.float32)

    dy = _get("dy", (B, T, N, V))
    dg = _get("dg", (B, T, N, V))
    dw = _get("dw", (N, V))
    ws_bytes = m2rnn_output_norm_backward_workspace_size(B, T, N, V)
    if ws_bytes == 0:
        raise M2RNNError(M2RNN_ERR_UNSUPPORTED, "m2rnn_output_norm_backward_workspace_size")
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    st = m2rnn_output_norm_backward(_ptr(y), _ptr(g), _ptr(w), _ptr(dout), float(eps), _ptr(dy), _ptr(dg),
                                    _ptr(dw), B, T, N, V, _dtype_code(g), _ptr(workspace), workspace.numel(),
                                    _stream_handle(stream))
    _check(st, "m2rnn_output_norm_backward")
    return dict(dy=dy, dg=dg, dw=dw)


def sync_status(workspace, stream=None):
    st, detail = m2rnn_sync_status(workspace.data_ptr(), _stream_handle(stream))
    return st, detail


def to_device(inp, device="cuda"):
    """Upload an ``inputs.M2RNNInputs`` batch: bf16 bit patterns become
    torch.bfloat16 tensors, float32 stays float32."""
    import numpy as np
    import torch
    res = {}
    for name, arr in inp.store.items():
        if arr.dtype == np.uint16:
            t = torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(arr))
        res[name] = t.to(device).contiguous()
    return res


def m2rnn_backward_noalloc(q, k, v, f, W, w_r, dy, dH_T, ckpt, ckpt_every, dq, dk, dv, df, dW,
                           dw_r, B, T, N, K, V, dtype, sync, stream) -> int:
    """The backward for callers that cannot allocate device memory: scratch
    comes from an array built into the library (see include/m2rnn.h for the
    limits).  Integers are device addresses, as for m2rnn_backward."""
    lib = load()
    fn = lib.m2rnn_backward_noalloc
    if fn.argtypes is None:
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        fn.restype = ci
        fn.argtypes = [vp] * 9 + [ci] + [vp] * 6 + [i64] * 5 + [ci, ci, vp]
    return fn(q, k, v, f, W, w_r, dy, dH_T, ckpt, ckpt_every, dq, dk, dv, df, dW, dw_r, B, T, N,
              K, V, dtype, sync, stream)


def m2rnn_backward_noalloc_status(stream):
    """Device-side status of the last allocation-free backward on the current
    device: returns (status, detail); synchronises `stream` first."""
    lib = load()
    fn = lib.m2rnn_backward_noalloc_status
    if fn.argtypes is None:
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    detail = ctypes.c_uint32(0)
    st = fn(stream, ctypes.byref(detail))
    return st, detail.value
