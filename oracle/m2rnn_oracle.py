"""Float64 CPU oracle for the M2RNN forward scan and its backward-through-time.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the test-suite, the smoke check of the package entry module and the
CPU-baseline leg of the benchmark call it.  It shares no code with the CUDA
library; both consume the same seeded inputs (float64 values of the stored
bf16/fp32 data).

Source: reading notes on "M2RNN: Non-Linear RNNs with Matrix-Valued States for
Scalable Language Modeling" (Mishra, Tan, Stoica, Gonzalez, Dao;
arXiv:2603.14360v2), section 2.1 (the paper's Eq. 10-12) for the forward and
section 2.7 (the notes' chain-rule correction of the paper's Algorithm 2) for
the backward.

Notation (per batch element b and head n, from H_0 = 0 unless an initial
state H_0 is given; the pages' fixed-size recurrent state is what lets a long
sequence be run in pieces, the state of one piece starting the next):
    Z_t = tanh(H_{t-1} W + k_t v_t^T)            (Eq. 10)
    H_t = f_t H_{t-1} + (1 - f_t) Z_t            (Eq. 11)
    y_t = H_t^T q_t + w_r * v_t                  (Eq. 12)
H, Z are K x V; W is V x V and multiplies from the right, so
(H W)_{ij} = sum_m H_{im} W_{mj}; q_t, k_t have K entries, v_t and w_r have V;
f_t is a scalar.  Array layouts: q, k [B,T,N,K]; v [B,T,N,V]; f [B,T,N];
W [N,V,V]; w_r [N,V]; y, dy [B,T,N,V]; H_0, dH_0, H_T, dH_T [B,N,K,V].

Multi-value sharing (section 2.4 of the notes): q and k may have a head
axis of length 1, [B,T,1,K], shared by every value head; each head keeps its
own v, f, W, w_r and state.  Their gradients are then summed over the heads
(section 2.7) and returned with the same [B,T,1,K] shape.

Every function is a plain loop over t, vectorised over (b, n) with numpy
matmul/einsum; there is no blocking, fusion or reordering beyond the equations.
"""
from __future__ import annotations

import numpy as np


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def _heads(q, k, v):
    """q, k broadcast to every value head (a shared q/k has a head axis of 1)."""
    N = v.shape[2]
    if q.shape[2] != N:
        if q.shape[2] != 1 or k.shape[2] != 1:
            raise ValueError("q/k need one head (shared) or as many heads as v")
        q = np.broadcast_to(q, q.shape[:2] + (N,) + q.shape[3:])
        k = np.broadcast_to(k, k.shape[:2] + (N,) + k.shape[3:])
    return q, k


def forward(q, k, v, f, W, w_r, return_states: bool = False, H_0=None):
    """M2RNN forward scan (Eq. 10-12) from H_0 (zero if None).

    Returns (y [B,T,N,V], H_T [B,N,K,V]); with ``return_states`` also the
    stacked H_t and Z_t, shape [T+1,B,N,K,V] (index 0 holds H_0) and
    [T,B,N,K,V] (index t-1 holds Z_t).
    """
    q, k, v, f, W, w_r = map(_as64, (q, k, v, f, W, w_r))
    q, k = _heads(q, k, v)
    B, T, N, K = q.shape
    V = v.shape[-1]
    H = np.zeros((B, N, K, V)) if H_0 is None else _as64(H_0).copy()
    y = np.empty((B, T, N, V))
    if return_states:
        Hs = np.empty((T + 1, B, N, K, V))
        Zs = np.empty((T, B, N, K, V))
        Hs[0] = H
    for t in range(T):
        kt, vt, qt = k[:, t], v[:, t], q[:, t]           # [B,N,K], [B,N,V], [B,N,K]
        ft = f[:, t][:, :, None, None]                    # [B,N,1,1]
        # Eq. 10: transform the old state by W (right multiplication), add the
        # rank-1 write k_t v_t^T, squash elementwise.
        A = np.matmul(H, W[None]) + kt[..., :, None] * vt[..., None, :]
        Z = np.tanh(A)
        # Eq. 11: gate blend between the retained and the candidate state.
        H = ft * H + (1.0 - ft) * Z
        # Eq. 12: read out along the K rows with q_t, plus the value residual.
        y[:, t] = np.einsum("bnkv,bnk->bnv", H, qt) + w_r[None] * vt
        if return_states:
            Hs[t + 1] = H
            Zs[t] = Z
    if return_states:
        return y, H, Hs, Zs
    return y, H


def backward(q, k, v, f, W, w_r, dy, dH_T=None, H_0=None, state_grad_clip=None):
    """Gradients of L = sum(dy * y) + <dH_T, H_T> with respect to every input
    (and to the initial state H_0, zero if None).

    ``state_grad_clip`` = c > 0 clips the recurrent state gradient at every
    step of BPTT (section 2.3 of the notes: training clips the per-step state
    gradient, separately from whole-model gradient clipping; the notes do not
    say how): each newly formed C_{t-1} is clamped elementwise to [-c, c]
    before it is used.  The results are then no longer the exact gradient.

    Follows the chain rule for Eq. 10-12 as derived in section 2.7 of the
    reading notes, with u_t the upstream gradient of the readout H_t^T q_t
    (equal to dy_t, since the value residual w_r*v_t enters y_t additively)
    and C_t the state gradient flowing back from steps after t (C_T = dH_T):
        R_t     = C_t + q_t u_t^T
        D_t     = ((1 - f_t) R_t) * (1 - Z_t * Z_t)
        C_{t-1} = f_t R_t + D_t W^T
        dq_t = H_t u_t          dk_t = D_t v_t
        dv_t = D_t^T k_t + w_r * u_t
        df_t = <R_t, H_{t-1} - Z_t>_F
        dW   = sum over b, t of H_{t-1}^T D_t
        dw_r = sum over b, t of u_t * v_t
    The value-residual terms (w_r * u_t in dv, and dw_r) are the direct-path
    contributions that the notes tell the reader to restore.

    The state gradient left after step 1, C_0, is dH_0 = dL/dH_0 (the same
    recursion carried one step further back).

    Returns a dict with dq, dk [B,T,N,K] ([B,T,1,K], summed over the heads,
    when q and k are shared); dv [B,T,N,V]; df [B,T,N]; dW [N,V,V];
    dw_r [N,V]; dH_0 [B,N,K,V]; all float64.
    """
    q, k, v, f, W, w_r, dy = map(_as64, (q, k, v, f, W, w_r, dy))
    shared = q.shape[2] != v.shape[2]
    q, k = _heads(q, k, v)
    B, T, N, K = q.shape
    V = v.shape[-1]
    _, _, Hs, Zs = forward(q, k, v, f, W, w_r, return_states=True, H_0=H_0)
    C = np.zeros((B, N, K, V)) if dH_T is None else _as64(dH_T).copy()
    dq = np.empty((B, T, N, K))
    dk = np.empty((B, T, N, K))
    dv = np.empty((B, T, N, V))
    df = np.empty((B, T, N))
    dW = np.zeros((N, V, V))
    dw_r = np.zeros((N, V))
    Wt = np.swapaxes(W, -1, -2)[None]                      # [1,N,V,V] = W^T
    for t in range(T - 1, -1, -1):
        u = dy[:, t]                                        # [B,N,V]
        qt, kt, vt = q[:, t], k[:, t], v[:, t]
        ft = f[:, t][:, :, None, None]
        H_prev, H_t, Z = Hs[t], Hs[t + 1], Zs[t]
        R = C + qt[..., :, None] * u[..., None, :]
        D = ((1.0 - ft) * R) * (1.0 - Z * Z)
        dq[:, t] = np.einsum("bnkv,bnv->bnk", H_t, u)
        dk[:, t] = np.einsum("bnkv,bnv->bnk", D, vt)
        dv[:, t] = np.einsum("bnkv,bnk->bnv", D, kt) + w_r[None] * u
        df[:, t] = np.einsum("bnkv,bnkv->bn", R, H_prev - Z)
        dW += np.einsum("bnkm,bnkj->nmj", H_prev, D)
        dw_r += np.einsum("bnv,bnv->nv", u, vt)
        C = ft * R + np.matmul(D, Wt)
        if state_grad_clip is not None and state_grad_clip > 0:
            C = np.clip(C, -state_grad_clip, state_grad_clip)
    if shared:  # one q/k for every head: their gradients sum over the heads
        dq = dq.sum(axis=2, keepdims=True)
        dk = dk.sum(axis=2, keepdims=True)
    return dict(dq=dq, dk=dk, dv=dv, df=df, dW=dW, dw_r=dw_r, dH_0=C)


def loss(q, k, v, f, W, w_r, dy, dH_T=None, H_0=None):
    """Scalar L = sum(dy * y) + <dH_T, H_T>, the function ``backward`` differentiates."""
    y, H_T = forward(q, k, v, f, W, w_r, H_0=H_0)
    val = float(np.sum(_as64(dy) * y))
    if dH_T is not None:
        val += float(np.sum(_as64(dH_T) * H_T))
    return val


# ---------------------------------------------------------------------------
# Input-dependent forget gate (section 2.2 of the notes, the paper's
# Eq. 13 and 17): f_{t,n} = (1 + exp(a_{t,n} + beta_n))^(-alpha_n)
#                         = exp(-alpha_n * softplus(a_{t,n} + beta_n)),
# alpha_n >= 0 keeps f in [0, 1]; alpha_n = 1 gives sigmoid(-a - beta).
# ---------------------------------------------------------------------------

def _softplus(x):
    return np.logaddexp(0.0, x)


def gate(a, alpha, beta):
    """f [B,T,N] from the gate pre-activation a [B,T,N] and per-head alpha, beta [N]."""
    a, alpha, beta = _as64(a), _as64(alpha), _as64(beta)
    return np.exp(-alpha * _softplus(a + beta))


def gate_backward(a, alpha, beta, df):
    """Chain rule through the gate: with s = softplus(a + beta) and
    ds/da = sigmoid(a + beta),
        da = df * f * (-alpha) * sigmoid(a + beta)
        dalpha = sum over b, t of df * f * (-s)
        dbeta  = sum over b, t of da
    Returns (da [B,T,N], dalpha [N], dbeta [N])."""
    a, alpha, beta, df = _as64(a), _as64(alpha), _as64(beta), _as64(df)
    x = a + beta
    f = np.exp(-alpha * _softplus(x))
    sig = 0.5 * (1.0 + np.tanh(0.5 * x))  # logistic function, overflow-free
    da = df * f * (-alpha) * sig
    dalpha = np.sum(df * f * (-_softplus(x)), axis=(0, 1))
    dbeta = np.sum(da, axis=(0, 1))
    return da, dalpha, dbeta


# ---------------------------------------------------------------------------
# Output path (section 2.3 of the notes, step 4): the readout is multiplied
# by the output gate g_t first, then RMS-normalised over the full width of a
# token, all heads together (Appendix C: the statistic spans every head's
# elements, d = N V), with a per-channel weight w [N,V]:
#     x = y * g,   s = (sum(x^2) / d + eps)^(-1/2),   out = w * x * s.
# The notes omit the stabilising epsilon; it is added inside the root here.
# Backward (Appendix C), with p = w * dout and r = sum(p * x):
#     dx = s p - r s^3 x / d,   dy = dx * g,   dg = dx * y,
#     dw = sum over b, t of dout * x * s.
# ---------------------------------------------------------------------------

def output_norm(y, g, w, eps=1e-6):
    """out [B,T,N,V] from y, g [B,T,N,V] and w [N,V]."""
    y, g, w = _as64(y), _as64(g), _as64(w)
    x = y * g
    d = x.shape[2] * x.shape[3]
    s = (np.sum(x * x, axis=(2, 3), keepdims=True) / d + eps) ** -0.5
    return w[None, None] * x * s


def output_norm_backward(y, g, w, dout, eps=1e-6):
    """Returns (dy, dg [B,T,N,V], dw [N,V])."""
    y, g, w, dout = _as64(y), _as64(g), _as64(w), _as64(dout)
    x = y * g
    d = x.shape[2] * x.shape[3]
    s = (np.sum(x * x, axis=(2, 3), keepdims=True) / d + eps) ** -0.5
    p = w[None, None] * dout
    r = np.sum(p * x, axis=(2, 3), keepdims=True)
    dx = s * p - r * s ** 3 * x / d
    return dx * g, dx * y, np.sum(dout * x * s, axis=(0, 1))
