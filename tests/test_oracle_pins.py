"""Pins of the float64 oracle against what the M2RNN pages and mathematics fix.

Each test ties the oracle to something other than itself: a library routine a
special case reduces to, a closed form, an invariant, or brute force.  Sources
are the reading notes on "M2RNN: Non-Linear RNNs with Matrix-Valued States for
Scalable Language Modeling": section 2.1 (Eq. 10-12 and the remarks after
them), section 1.2 (row independence), section 2.5 (Theorem 1 / Appendix B,
Eq. 25), section 2.6 (independent (b, n) work units) and section 2.7 (the
chain-rule backward).
"""
import numpy as np
import pytest
import torch

from matrix_state_non_gb300.inputs import make_inputs
from oracle import backward, forward, loss

NAMES = ("q", "k", "v", "f", "W", "w_r")


def _args(inp):
    return [inp.exact[n] for n in NAMES]


def _rand(B=2, N=3, T=7, K=5, V=4, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, N, K)) / np.sqrt(K)
    k = rng.standard_normal((B, T, N, K)) / np.sqrt(K)
    v = rng.standard_normal((B, T, N, V))
    f = 1.0 / (1.0 + np.exp(-(rng.standard_normal((B, T, N)) + 2.0)))
    W = rng.standard_normal((N, V, V)) / np.sqrt(V)
    w_r = rng.standard_normal((N, V))
    return q, k, v, f, W, w_r


# --------------------------------------------------------------------------
# Forward pins
# --------------------------------------------------------------------------

@pytest.mark.parametrize("V,T", [(4, 9), (16, 33)])
def test_theorem1_reduces_to_torch_tanh_rnn(V, T):
    """Theorem 1 (section 2.5): f=0, w_r=0, q=k=e_1 turns row 1 of H into the
    vanilla tanh RNN h_t = tanh(W^T h_{t-1} + v_t) and leaves rows 2..K at 0.
    torch.nn.RNN computes h_t = tanh(x_t W_ih^T + h_{t-1} W_hh^T), so
    W_ih = I and W_hh = W^T give the same recurrence in row form."""
    rng = np.random.default_rng(7)
    B, N, K = 2, 3, 5
    W = rng.standard_normal((N, V, V)) / np.sqrt(V) * 1.5
    v = rng.standard_normal((B, T, N, V))
    e1 = np.zeros(K)
    e1[0] = 1.0
    q = np.broadcast_to(e1, (B, T, N, K)).copy()
    k = q.copy()
    f = np.zeros((B, T, N))
    w_r = np.zeros((N, V))
    y, H_T = forward(q, k, v, f, W, w_r)
    for n in range(N):
        rnn = torch.nn.RNN(V, V, nonlinearity="tanh", bias=False, batch_first=True).double()
        with torch.no_grad():
            rnn.weight_ih_l0.copy_(torch.eye(V, dtype=torch.float64))
            rnn.weight_hh_l0.copy_(torch.from_numpy(W[n].T.copy()))
            out, h_last = rnn(torch.from_numpy(v[:, :, n].copy()))
        np.testing.assert_allclose(y[:, :, n], out.numpy(), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(H_T[:, n, 0], h_last[0].numpy(), rtol=1e-12, atol=1e-13)
    assert np.all(H_T[:, :, 1:, :] == 0.0)


def test_single_step_closed_form():
    """T=1 from H_0=0 (Eq. 10-12): H_1 = (1-f_1) tanh(k_1 v_1^T),
    y_1 = H_1^T q_1 + w_r * v_1."""
    q, k, v, f, W, w_r = _rand(T=1)
    y, H_T = forward(q, k, v, f, W, w_r)
    B, _, N, K = q.shape
    for b in range(B):
        for n in range(N):
            H1 = (1.0 - f[b, 0, n]) * np.tanh(np.outer(k[b, 0, n], v[b, 0, n]))
            np.testing.assert_allclose(H_T[b, n], H1, rtol=1e-14, atol=1e-15)
            np.testing.assert_allclose(y[b, 0, n], H1.T @ q[b, 0, n] + w_r[n] * v[b, 0, n],
                                       rtol=1e-13, atol=1e-14)


def test_forget_zero_without_transition_is_memoryless():
    """f=0 and W=0: the candidate has no history term, so H_t = tanh(k_t v_t^T)
    at every step (Eq. 10-11 with the retain branch and H W removed)."""
    q, k, v, f, W, w_r = _rand(T=6)
    f = np.zeros_like(f)
    W = np.zeros_like(W)
    y, H_T = forward(q, k, v, f, W, w_r)
    B, T, N, K = q.shape
    for b in range(B):
        for t in range(T):
            for n in range(N):
                Ht = np.tanh(np.outer(k[b, t, n], v[b, t, n]))
                np.testing.assert_allclose(y[b, t, n], Ht.T @ q[b, t, n] + w_r[n] * v[b, t, n],
                                           rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(H_T, np.tanh(k[:, -1, :, :, None] * v[:, -1, :, None, :]),
                               rtol=1e-14, atol=1e-15)


def test_forget_one_keeps_state():
    """f=1 keeps the state (section 2.1 remark): from H_0=0 the state stays 0
    and the readout is exactly the value residual w_r * v_t."""
    inp = make_inputs(2, 3, 11, 8, 4, "bf16", seed=3, f_mode="ones")
    y, H_T = forward(*_args(inp))
    assert np.all(H_T == 0.0)
    np.testing.assert_array_equal(y, inp.exact["w_r"][None, None] * inp.exact["v"])


def test_forget_one_after_t0_freezes_state():
    """f_t = 1 for t > t0 leaves H_T equal to H_{t0} (retain branch only)."""
    q, k, v, f, W, w_r = _rand(T=9)
    t0 = 4
    f2 = f.copy()
    f2[:, t0:] = 1.0
    _, H_T = forward(q, k, v, f2, W, w_r)
    _, H_t0 = forward(q[:, :t0], k[:, :t0], v[:, :t0], f[:, :t0], W, w_r)
    np.testing.assert_array_equal(H_T, H_t0)


def test_state_is_bounded():
    """f in [0,1] and H_0 = 0 make every H_t a convex combination of bounded
    values, so |H_ij| <= 1 (section 2.1), even for huge writes."""
    q, k, v, f, W, w_r = _rand(T=40, K=6, V=5, seed=5)
    k = k * 50.0
    v = v * 50.0
    W = W * 20.0
    f = np.random.default_rng(1).uniform(0.0, 1.0, size=f.shape)
    _, _, Hs, Zs = forward(q, k, v, f, W, w_r, return_states=True)
    assert np.all(np.abs(Hs) <= 1.0)
    assert np.all(np.abs(Zs) <= 1.0)


def test_key_rows_are_independent_and_permutation_equivariant():
    """W mixes value columns only; key rows never mix (section 1.2).  Permuting
    the K entries of q and k together permutes the rows of H_T and leaves y
    unchanged."""
    q, k, v, f, W, w_r = _rand(K=7, seed=11)
    perm = np.random.default_rng(2).permutation(q.shape[-1])
    y, H_T = forward(q, k, v, f, W, w_r)
    y2, H_T2 = forward(q[..., perm], k[..., perm], v, f, W, w_r)
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(H_T2, H_T[:, :, perm, :])


def test_chains_are_independent():
    """Each (b, n) pair is its own work unit (section 2.6): running one chain
    alone gives the same numbers as the batched run."""
    q, k, v, f, W, w_r = _rand(B=3, N=2, seed=4)
    y, H_T = forward(q, k, v, f, W, w_r)
    for b in range(3):
        for n in range(2):
            sl = (slice(b, b + 1), slice(None), slice(n, n + 1))
            y1, H1 = forward(q[sl], k[sl], v[sl], f[sl], W[n:n + 1], w_r[n:n + 1])
            np.testing.assert_array_equal(y1[0, :, 0], y[b, :, n])
            np.testing.assert_array_equal(H1[0, 0], H_T[b, n])


def test_identity_transition_is_elementwise_scalar_recurrence():
    """W = I (the paper's initialisation) makes H W = H, so every element runs
    its own scalar recurrence h <- f h + (1-f) tanh(h + k_i v_j)."""
    q, k, v, f, W, w_r = _rand(B=1, N=2, T=12, K=3, V=4, seed=8)
    W = np.broadcast_to(np.eye(4), W.shape).copy()
    y, H_T = forward(q, k, v, f, W, w_r)
    B, T, N, K = q.shape
    V = v.shape[-1]
    for n in range(N):
        h = np.zeros((K, V))
        for t in range(T):
            ft = f[0, t, n]
            for i in range(K):
                for j in range(V):
                    h[i, j] = ft * h[i, j] + (1.0 - ft) * np.tanh(h[i, j] + k[0, t, n, i] * v[0, t, n, j])
            yt = [sum(q[0, t, n, i] * h[i, j] for i in range(K)) + w_r[n, j] * v[0, t, n, j]
                  for j in range(V)]
            np.testing.assert_allclose(y[0, t, n], yt, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(H_T[0, n], h, rtol=1e-14, atol=1e-15)


# --------------------------------------------------------------------------
# Backward pins
# --------------------------------------------------------------------------

def _fd_grads(args, dy, dH_T, eps=1e-6):
    grads = []
    for idx in range(6):
        x = args[idx]
        g = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            xp = [a.copy() for a in args]
            xm = [a.copy() for a in args]
            xp[idx][mi] += eps
            xm[idx][mi] -= eps
            g[mi] = (loss(*xp, dy, dH_T) - loss(*xm, dy, dH_T)) / (2 * eps)
        grads.append(g)
    return dict(zip(("dq", "dk", "dv", "df", "dW", "dw_r"), grads))


@pytest.mark.parametrize("B,N,T,K,V,with_dH", [
    (1, 1, 1, 2, 3, False), (1, 1, 2, 3, 2, True), (1, 1, 5, 4, 3, True),
    (2, 2, 4, 3, 4, True), (2, 1, 5, 2, 2, False),
])
def test_backward_matches_central_finite_differences(B, N, T, K, V, with_dH):
    """Brute force: central differences of L = sum(dy*y) + <dH_T, H_T> in
    float64 over every input element.  The notes (section 2.7) warn that the
    paper's Algorithm 2 is wrong as printed, so the hand-derived backward is
    checked against the definition of the derivative itself."""
    args = list(_rand(B, N, T, K, V, seed=100 + T + K))
    rng = np.random.default_rng(9)
    dy = rng.standard_normal((B, T, N, V))
    dH_T = rng.standard_normal((B, N, K, V)) if with_dH else None
    g = backward(*args, dy, dH_T)
    fd = _fd_grads(args, dy, dH_T)
    for name in fd:
        np.testing.assert_allclose(g[name], fd[name], rtol=2e-7, atol=2e-8, err_msg=name)


def _torch_forward(q, k, v, f, W, w_r, H_0=None):
    """An independent restatement of Eq. 10-12 in torch, written with explicit
    per-row loops over the key index so it shares no structure with the
    vectorised oracle."""
    B, T, N, K = q.shape
    ys = []
    H = [[[torch.zeros(v.shape[-1], dtype=torch.float64) if H_0 is None else H_0[b, n, i]
           for i in range(K)] for n in range(N)] for b in range(B)]
    for t in range(T):
        yt_b = []
        for b in range(B):
            yt_n = []
            for n in range(N):
                rows = []
                for i in range(K):
                    z = torch.tanh(H[b][n][i] @ W[n] + k[b, t, n, i] * v[b, t, n])
                    rows.append(f[b, t, n] * H[b][n][i] + (1 - f[b, t, n]) * z)
                H[b][n] = rows
                yt_n.append(sum(q[b, t, n, i] * rows[i] for i in range(K)) + w_r[n] * v[b, t, n])
            yt_b.append(torch.stack(yt_n))
        ys.append(torch.stack(yt_b))
    y = torch.stack(ys, dim=1)
    H_T = torch.stack([torch.stack([torch.stack(H[b][n]) for n in range(N)]) for b in range(B)])
    return y, H_T


def test_backward_matches_torch_autograd():
    """torch.autograd (float64) through an independently written forward."""
    args = _rand(B=2, N=2, T=6, K=4, V=3, seed=21)
    rng = np.random.default_rng(3)
    dy = rng.standard_normal((2, 6, 2, 3))
    dH_T = rng.standard_normal((2, 2, 4, 3))
    ts = [torch.tensor(a, requires_grad=True) for a in args]
    y, H_T = _torch_forward(*ts)
    y_np, H_np = forward(*args)
    np.testing.assert_allclose(y.detach().numpy(), y_np, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(H_T.detach().numpy(), H_np, rtol=1e-12, atol=1e-13)
    L = (y * torch.from_numpy(dy)).sum() + (H_T * torch.from_numpy(dH_T)).sum()
    L.backward()
    g = backward(*args, dy, dH_T)
    for name, t in zip(("dq", "dk", "dv", "df", "dW", "dw_r"), ts):
        np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)


def test_backward_forget_one_closed_form():
    """f = 1: H stays 0 and D = 0 (its (1-f) factor vanishes), so dq = dk = 0,
    dW = 0, dv = w_r * u, dw_r = sum u*v, C_{t-1} = R_t, hence
    R_t = dH_T + sum_{s>=t} q_s u_s^T and df_t = <R_t, 0 - tanh(k_t v_t^T)>."""
    q, k, v, f, W, w_r = _rand(B=2, N=2, T=5, K=3, V=4, seed=31)
    f = np.ones_like(f)
    rng = np.random.default_rng(5)
    dy = rng.standard_normal(v.shape)
    dH_T = rng.standard_normal((2, 2, 3, 4))
    g = backward(q, k, v, f, W, w_r, dy, dH_T)
    assert np.all(g["dq"] == 0) and np.all(g["dk"] == 0) and np.all(g["dW"] == 0)
    np.testing.assert_allclose(g["dv"], w_r[None, None] * dy, rtol=1e-15)
    np.testing.assert_allclose(g["dw_r"], np.einsum("btnv,btnv->nv", dy, v), rtol=1e-13)
    B, T, N, K = q.shape
    for b in range(B):
        for n in range(N):
            R = dH_T[b, n].copy()
            for t in range(T - 1, -1, -1):
                R = R + np.outer(q[b, t, n], dy[b, t, n])
                expect = -np.sum(R * np.tanh(np.outer(k[b, t, n], v[b, t, n])))
                np.testing.assert_allclose(g["df"][b, t, n], expect, rtol=1e-12, atol=1e-13)


def test_backward_single_step_by_hand():
    """T=1 by hand: H_1 = (1-f) Z, Z = tanh(k v^T).  dL/dH_1 = q u^T + dH_T;
    through Z: (1-f)(dL/dH_1)(1-Z^2) w.r.t. the pre-activation k v^T, whence
    dk = that v, dv = that^T k + w_r u; df = -<dL/dH_1, Z>; dW = H_0^T(.) = 0."""
    q, k, v, f, W, w_r = _rand(B=1, N=1, T=1, K=3, V=2, seed=41)
    rng = np.random.default_rng(6)
    dy = rng.standard_normal(v.shape)
    dH = rng.standard_normal((1, 1, 3, 2))
    g = backward(q, k, v, f, W, w_r, dy, dH)
    qq, kk, vv, ff, u = q[0, 0, 0], k[0, 0, 0], v[0, 0, 0], f[0, 0, 0], dy[0, 0, 0]
    Z = np.tanh(np.outer(kk, vv))
    H1 = (1 - ff) * Z
    G = np.outer(qq, u) + dH[0, 0]
    P = (1 - ff) * G * (1 - Z ** 2)
    np.testing.assert_allclose(g["dq"][0, 0, 0], H1 @ u, rtol=1e-13)
    np.testing.assert_allclose(g["dk"][0, 0, 0], P @ vv, rtol=1e-13)
    np.testing.assert_allclose(g["dv"][0, 0, 0], P.T @ kk + w_r[0] * u, rtol=1e-13)
    np.testing.assert_allclose(g["df"][0, 0, 0], -np.sum(G * Z), rtol=1e-13)
    assert np.all(g["dW"] == 0)
    np.testing.assert_allclose(g["dw_r"][0], u * vv, rtol=1e-15)


def _mutant_forward(mode):
    """A copy of Eq. 10-12 with one planted mistake (test-only, CPU)."""
    def fwd(q, k, v, f, W, w_r):
        B, T, N, K = q.shape
        V = v.shape[-1]
        H = np.zeros((B, N, K, V))
        y = np.empty((B, T, N, V))
        Wm = np.swapaxes(W, -1, -2) if mode == "transpose_W" else W
        for t in range(T):
            sign = -1.0 if mode == "minus_write" else 1.0
            Z = np.tanh(np.matmul(H, Wm[None]) + sign * k[:, t][..., :, None] * v[:, t][..., None, :])
            ft = f[:, t][:, :, None, None]
            H = (1 - ft) * H + ft * Z if mode == "swap_blend" else ft * H + (1 - ft) * Z
            res = 0.0 if mode == "no_residual" else w_r[None] * v[:, t]
            if mode == "read_columns":
                y[:, t] = np.einsum("bnkv,bnv->bnk", H, q[:, t][..., :V]) + res
            else:
                y[:, t] = np.einsum("bnkv,bnk->bnv", H, q[:, t]) + res
        return y, H
    return fwd


def _pins_pass(fwd):
    """Run the forward pins above with ``forward`` replaced by ``fwd``."""
    global forward
    saved = forward
    forward = fwd
    try:
        test_theorem1_reduces_to_torch_tanh_rnn(4, 9)
        test_single_step_closed_form()
        test_forget_zero_without_transition_is_memoryless()
        test_forget_one_keeps_state()
        return True
    except (AssertionError, ValueError):
        return False
    finally:
        forward = saved


@pytest.mark.parametrize("mode", ["transpose_W", "minus_write", "swap_blend",
                                  "no_residual", "read_columns"])
def test_planted_mistakes_fail_a_pin(mode):
    """Plausible mistakes (transposed W, wrong sign of the write, swapped gate
    blend, dropped value residual, readout over the wrong axis) each fail at
    least one forward pin, while the oracle itself passes them all."""
    assert _pins_pass(forward)
    assert not _pins_pass(_mutant_forward(mode))


# --------------------------------------------------------------------------
# Initial state H_0 and its gradient (running a sequence in pieces)
# --------------------------------------------------------------------------

def test_forward_pieces_compose_exactly():
    """The state is the whole memory: the forward over [0, T) equals the
    forward over [0, T1) followed by the forward over [T1, T) started from
    the first piece's final state (the same float64 operations in the same
    order, so bit for bit)."""
    args = _rand(B=2, N=2, T=11, K=4, V=3, seed=51)
    y, H_T = forward(*args)
    for T1 in (1, 4, 10):
        a1 = [a[:, :T1] if a.ndim >= 3 else a for a in args[:4]] + list(args[4:])
        a2 = [a[:, T1:] if a.ndim >= 3 else a for a in args[:4]] + list(args[4:])
        y1, H1 = forward(*a1)
        y2, H2 = forward(*a2, H_0=H1)
        np.testing.assert_array_equal(np.concatenate([y1, y2], axis=1), y)
        np.testing.assert_array_equal(H2, H_T)


def test_backward_pieces_compose():
    """Backward in two pieces: the later piece (started from H_{T1}, with the
    upstream dH_T) returns dH_0, which is the upstream state gradient of the
    earlier piece; per-step gradients concatenate and dW, dw_r add up to the
    single-pass result."""
    args = _rand(B=2, N=2, T=9, K=3, V=4, seed=52)
    rng = np.random.default_rng(8)
    dy = rng.standard_normal((2, 9, 2, 4))
    dH_T = rng.standard_normal((2, 2, 3, 4))
    H_0 = 0.5 * rng.standard_normal((2, 2, 3, 4))
    g = backward(*args, dy, dH_T, H_0=H_0)
    T1 = 4
    a1 = [a[:, :T1] if a.ndim >= 3 else a for a in args[:4]] + list(args[4:])
    a2 = [a[:, T1:] if a.ndim >= 3 else a for a in args[:4]] + list(args[4:])
    _, H1 = forward(*a1, H_0=H_0)
    g2 = backward(*a2, dy[:, T1:], dH_T, H_0=H1)
    g1 = backward(*a1, dy[:, :T1], g2["dH_0"], H_0=H_0)
    for name in ("dq", "dk", "dv", "df"):
        np.testing.assert_allclose(np.concatenate([g1[name], g2[name]], axis=1), g[name], rtol=1e-12, atol=1e-13)
    for name in ("dW", "dw_r"):
        np.testing.assert_allclose(g1[name] + g2[name], g[name], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g1["dH_0"], g["dH_0"], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("B,N,T,K,V", [(1, 1, 1, 2, 3), (1, 1, 4, 3, 2), (2, 2, 3, 2, 3)])
def test_initial_state_gradient_matches_finite_differences(B, N, T, K, V):
    """Brute force on H_0: central differences of L over every element of H_0,
    and the other inputs' gradients stay right with a non-zero H_0."""
    args = list(_rand(B, N, T, K, V, seed=200 + T + K))
    rng = np.random.default_rng(11)
    dy = rng.standard_normal((B, T, N, V))
    dH_T = rng.standard_normal((B, N, K, V))
    H_0 = rng.standard_normal((B, N, K, V))
    g = backward(*args, dy, dH_T, H_0=H_0)
    eps = 1e-6
    fd = np.zeros_like(H_0)
    it = np.nditer(H_0, flags=["multi_index"])
    for _ in it:
        mi = it.multi_index
        hp, hm = H_0.copy(), H_0.copy()
        hp[mi] += eps
        hm[mi] -= eps
        fd[mi] = (loss(*args, dy, dH_T, H_0=hp) - loss(*args, dy, dH_T, H_0=hm)) / (2 * eps)
    np.testing.assert_allclose(g["dH_0"], fd, rtol=2e-7, atol=2e-8)
    x = args[4]  # W, whose gradient runs through H_{t-1} and so sees H_0
    fdw = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        mi = it.multi_index
        xp = [a.copy() for a in args]
        xm = [a.copy() for a in args]
        xp[4][mi] += eps
        xm[4][mi] -= eps
        fdw[mi] = (loss(*xp, dy, dH_T, H_0=H_0) - loss(*xm, dy, dH_T, H_0=H_0)) / (2 * eps)
    np.testing.assert_allclose(g["dW"], fdw, rtol=2e-7, atol=2e-8)


def test_initial_state_forget_one_closed_form():
    """f = 1 from a non-zero H_0: the state never moves (H_t = H_0), so
    y_t = H_0^T q_t + w_r v_t; D = 0, C_{t-1} = R_t, hence
    dH_0 = dH_T + sum_t q_t u_t^T, dq_t = H_0 u_t, dW = 0."""
    q, k, v, f, W, w_r = _rand(B=2, N=2, T=5, K=3, V=4, seed=53)
    f = np.ones_like(f)
    rng = np.random.default_rng(12)
    H_0 = rng.standard_normal((2, 2, 3, 4))
    dy = rng.standard_normal(v.shape)
    dH_T = rng.standard_normal((2, 2, 3, 4))
    y, H_T = forward(q, k, v, f, W, w_r, H_0=H_0)
    np.testing.assert_array_equal(H_T, H_0)
    np.testing.assert_allclose(y, np.einsum("bnkv,btnk->btnv", H_0, q) + w_r[None, None] * v, rtol=1e-13)
    g = backward(q, k, v, f, W, w_r, dy, dH_T, H_0=H_0)
    np.testing.assert_allclose(g["dH_0"], dH_T + np.einsum("btnk,btnv->bnkv", q, dy), rtol=1e-13)
    np.testing.assert_allclose(g["dq"], np.einsum("bnkv,btnv->btnk", H_0, dy), rtol=1e-13)
    assert np.all(g["dW"] == 0)


def test_initial_state_gradient_matches_torch_autograd():
    """torch.autograd through the independently written forward, H_0 a leaf."""
    args = _rand(B=1, N=2, T=5, K=3, V=4, seed=54)
    rng = np.random.default_rng(13)
    H_0 = rng.standard_normal((1, 2, 3, 4))
    dy = rng.standard_normal((1, 5, 2, 4))
    dH_T = rng.standard_normal((1, 2, 3, 4))
    ts = [torch.tensor(a) for a in args]
    h0 = torch.tensor(H_0, requires_grad=True)
    y, H_T = _torch_forward(*ts, H_0=h0)
    L = (y * torch.from_numpy(dy)).sum() + (H_T * torch.from_numpy(dH_T)).sum()
    L.backward()
    g = backward(*args, dy, dH_T, H_0=H_0)
    np.testing.assert_allclose(g["dH_0"], h0.grad.numpy(), rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------
# Multi-value heads: one q/k shared by every value head
# --------------------------------------------------------------------------

def _shared_qk(B=2, N=3, T=6, K=4, V=3, seed=60):
    q, k, v, f, W, w_r = _rand(B, N, T, K, V, seed)
    return q[:, :, :1].copy(), k[:, :, :1].copy(), v, f, W, w_r


def test_shared_qk_equals_replicated_heads():
    """A shared q/k is the multi-head case with the same q/k in every head
    (section 2.4): the forward is identical, and the shared gradients are the
    per-head gradients summed over heads (section 2.7)."""
    q1, k1, v, f, W, w_r = _shared_qk()
    N = v.shape[2]
    qN, kN = np.repeat(q1, N, axis=2), np.repeat(k1, N, axis=2)
    y1, H1 = forward(q1, k1, v, f, W, w_r)
    yN, HN = forward(qN, kN, v, f, W, w_r)
    np.testing.assert_array_equal(y1, yN)
    np.testing.assert_array_equal(H1, HN)
    rng = np.random.default_rng(14)
    dy = rng.standard_normal(v.shape)
    g1 = backward(q1, k1, v, f, W, w_r, dy)
    gN = backward(qN, kN, v, f, W, w_r, dy)
    assert g1["dq"].shape == q1.shape and g1["dk"].shape == k1.shape
    np.testing.assert_allclose(g1["dq"], gN["dq"].sum(axis=2, keepdims=True), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(g1["dk"], gN["dk"].sum(axis=2, keepdims=True), rtol=1e-13, atol=1e-15)
    for name in ("dv", "df", "dW", "dw_r", "dH_0"):
        np.testing.assert_array_equal(g1[name], gN[name])


def test_shared_qk_gradient_matches_finite_differences():
    """Brute force on the shared q and k (one key/query vector feeding every head)."""
    q1, k1, v, f, W, w_r = _shared_qk(B=1, N=3, T=4, K=3, V=2, seed=61)
    rng = np.random.default_rng(15)
    dy = rng.standard_normal(v.shape)
    args = [q1, k1, v, f, W, w_r]
    g = backward(*args, dy)
    eps = 1e-6
    for idx, name in ((0, "dq"), (1, "dk")):
        fd = np.zeros_like(args[idx])
        it = np.nditer(args[idx], flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            xp = [a.copy() for a in args]
            xm = [a.copy() for a in args]
            xp[idx][mi] += eps
            xm[idx][mi] -= eps
            fd[mi] = (loss(*xp, dy) - loss(*xm, dy)) / (2 * eps)
        np.testing.assert_allclose(g[name], fd, rtol=2e-7, atol=2e-8, err_msg=name)


# --------------------------------------------------------------------------
# Per-step clipping of the recurrent state gradient (not an exact gradient)
# --------------------------------------------------------------------------

def test_state_grad_clip_large_is_exact_gradient():
    args = _rand(B=2, N=2, T=7, K=3, V=4, seed=70)
    dy = np.random.default_rng(16).standard_normal((2, 7, 2, 4))
    g0 = backward(*args, dy)
    g1 = backward(*args, dy, state_grad_clip=1e30)
    for name in g0:
        np.testing.assert_array_equal(g0[name], g1[name])


def test_state_grad_clip_forget_one_by_hand():
    """f = 1: D = 0, so C_{t-1} = clamp(C_t + q_t u_t^T) -- a clamped running
    sum computed here by hand -- and dH_0 is its last value, dq_t = H_t u_t
    with H_t = 0 (no input reaches the state), df_t = <R_t, -Z_t>."""
    q, k, v, f, W, w_r = _rand(B=1, N=1, T=6, K=3, V=4, seed=71)
    f = np.ones_like(f)
    rng = np.random.default_rng(17)
    dy = 3.0 * rng.standard_normal(v.shape)
    dH_T = rng.standard_normal((1, 1, 3, 4))
    c = 0.7
    g = backward(q, k, v, f, W, w_r, dy, dH_T, state_grad_clip=c)
    C = dH_T[0, 0].copy()
    for t in range(5, -1, -1):
        R = C + np.outer(q[0, t, 0], dy[0, t, 0])
        np.testing.assert_allclose(g["df"][0, t, 0], -np.sum(R * np.tanh(np.outer(k[0, t, 0], v[0, t, 0]))),
                                   rtol=1e-12, atol=1e-13)
        C = np.minimum(np.maximum(R, -c), c)
    np.testing.assert_allclose(g["dH_0"][0, 0], C, rtol=1e-13)
    assert np.all(np.abs(g["dH_0"]) <= c)


def test_state_grad_clip_bounds_every_state_gradient():
    """With clipping, every C_t handed to the next step lies in [-c, c]: the
    dq it produces (H_t u_t uses no C) is unchanged, while dH_0 is bounded."""
    args = _rand(B=2, N=2, T=9, K=4, V=3, seed=72)
    dy = 5.0 * np.random.default_rng(18).standard_normal((2, 9, 2, 3))
    g0 = backward(*args, dy)
    g1 = backward(*args, dy, state_grad_clip=0.05)
    np.testing.assert_array_equal(g0["dq"], g1["dq"])
    assert np.all(np.abs(g1["dH_0"]) <= 0.05)
    assert not np.allclose(g0["dk"], g1["dk"])


# --------------------------------------------------------------------------
# The forget gate f = exp(-alpha softplus(a + beta)) (section 2.2)
# --------------------------------------------------------------------------

from oracle import gate, gate_backward  # noqa: E402


def _gate_args(B=2, T=5, N=3, seed=80):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, T, N)) * 2.0, rng.uniform(0.1, 2.0, N), rng.standard_normal(N)


def test_gate_alpha_one_is_a_sigmoid():
    """alpha = 1: f = (1 + e^{a+beta})^{-1} = sigmoid(-a - beta) (section 2.2)."""
    a, _, beta = _gate_args()
    f = gate(a, np.ones_like(beta), beta)
    np.testing.assert_allclose(f, 1.0 / (1.0 + np.exp(a + beta)), rtol=1e-13)
    assert np.all((f >= 0) & (f <= 1))


def test_gate_power_form():
    """The two printed forms agree: (1 + e^{a+beta})^{-alpha}."""
    a, alpha, beta = _gate_args(seed=81)
    np.testing.assert_allclose(gate(a, alpha, beta), (1.0 + np.exp(a + beta)) ** (-alpha), rtol=1e-12)


def test_gated_scan_gradient_matches_finite_differences():
    """Through the gate and the scan: central differences of the loss with
    f = gate(a, alpha, beta) with respect to a, alpha and beta."""
    q, k, v, _, W, w_r = _rand(B=1, N=2, T=4, K=3, V=2, seed=82)
    a, alpha, beta = _gate_args(B=1, T=4, N=2, seed=83)
    dy = np.random.default_rng(19).standard_normal(v.shape)

    def L(a_, al_, be_):
        return loss(q, k, v, gate(a_, al_, be_), W, w_r, dy)

    df = backward(q, k, v, gate(a, alpha, beta), W, w_r, dy)["df"]
    da, dal, dbe = gate_backward(a, alpha, beta, df)
    eps = 1e-6
    for x, g_an, name in ((a, da, "a"), (alpha, dal, "alpha"), (beta, dbe, "beta")):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[mi] += eps
            xm[mi] -= eps
            args_p = [xp if y is x else y for y in (a, alpha, beta)]
            args_m = [xm if y is x else y for y in (a, alpha, beta)]
            fd[mi] = (L(*args_p) - L(*args_m)) / (2 * eps)
        np.testing.assert_allclose(g_an, fd, rtol=2e-7, atol=2e-8, err_msg=name)


# --------------------------------------------------------------------------
# Output gate and RMSNorm over the full width (section 2.3, Appendix C)
# --------------------------------------------------------------------------

from oracle import output_norm, output_norm_backward  # noqa: E402


def test_output_norm_is_torch_rms_norm():
    """Reduces to a library routine: torch's RMSNorm over the last N*V values
    of y * g, with the per-channel weight, forward and autograd backward."""
    rng = np.random.default_rng(90)
    B, T, N, V = 2, 3, 4, 5
    y, g = rng.standard_normal((B, T, N, V)), rng.standard_normal((B, T, N, V))
    w, dout = rng.standard_normal((N, V)), rng.standard_normal((B, T, N, V))
    eps = 1e-5
    ty, tg, tw = (torch.tensor(x, requires_grad=True) for x in (y, g, w))
    tout = torch.nn.functional.rms_norm((ty * tg).reshape(B, T, N * V), (N * V,), tw.reshape(N * V), eps)
    np.testing.assert_allclose(output_norm(y, g, w, eps), tout.detach().numpy().reshape(B, T, N, V), rtol=1e-12)
    (tout * torch.from_numpy(dout).reshape(B, T, N * V)).sum().backward()
    dy, dg, dw = output_norm_backward(y, g, w, dout, eps)
    np.testing.assert_allclose(dy, ty.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, tg.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dw, tw.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_output_norm_scale_invariance():
    """With eps = 0 the output does not change when y is scaled (and is
    unit-RMS before the weight)."""
    rng = np.random.default_rng(91)
    y, g = rng.standard_normal((1, 2, 3, 4)), rng.standard_normal((1, 2, 3, 4))
    w = np.ones((3, 4))
    o1 = output_norm(y, g, w, eps=0.0)
    np.testing.assert_allclose(output_norm(7.5 * y, g, w, eps=0.0), o1, rtol=1e-13)
    np.testing.assert_allclose(np.mean(o1 ** 2, axis=(2, 3)), 1.0, rtol=1e-13)
