"""GPU parity for the fused forget gate and the gated RMSNorm output path
(reading notes, sections 2.2 and 2.3, Appendix C).

The gate f = exp(-alpha softplus(a + beta)) is computed inside every scan
kernel family; its backward turns df into da, dalpha, dbeta.  The output path
normalises y * g over each token's N V elements.  Everything is compared
element by element with the float64 oracle on the same seeded inputs.
"""
import numpy as np
import pytest

from matrix_state_non_gb300.inputs import make_gate_inputs, make_inputs, make_norm_inputs
from oracle import backward as oracle_backward
from oracle import forward as oracle_forward
from oracle import gate, gate_backward, output_norm, output_norm_backward
from parity_util import TOL_BF16_MAXABS_Y, TOL_BF16_REL, TOL_F32, max_abs, rel_fro

pytestmark = pytest.mark.gpu


def _dev(arr):
    import torch
    if arr.dtype == np.uint16:
        t = torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.cuda().contiguous()


def _gated_case(B, N, T, K, V, dtype, seed, shared_qk=False):
    inp = make_inputs(B, N, T, K, V, dtype, seed=seed, with_dy=True)
    gs, ge = make_gate_inputs(B, T, N, dtype, seed=seed + 1)
    if shared_qk:
        for name in ("q", "k"):
            inp.store[name] = np.ascontiguousarray(inp.store[name][:, :, :1])
            inp.exact[name] = np.ascontiguousarray(inp.exact[name][:, :, :1])
    return inp, gs, ge


def _oracle_gated_args(inp, ge):
    e = inp.exact
    q, k = e["q"], e["k"]
    return [q, k, e["v"], gate(ge["a"], ge["alpha"], ge["beta"]), e["W"], e["w_r"]]


def _run_gated(inp, gs, backward=False, ckpt_every=14, reuse=False, stash=False):
    import torch
    from matrix_state_non_gb300 import binding
    d = {n: _dev(x) for n, x in inp.store.items()}
    g = tuple(_dev(gs[n]) for n in ("a", "alpha", "beta"))
    args = (d["q"], d["k"], d["v"], None, d["W"], d["w_r"])
    if not backward:
        out = binding.forward(*args, gate=g, ckpt_every=ckpt_every)
        st, detail = binding.sync_status(out["workspace"])
        assert st == binding.M2RNN_OK, (binding.status_string(st), detail)
        torch.cuda.synchronize()
        return {n: out[n].cpu().numpy() for n in ("y", "H_T")}
    ckpt = z = None
    if reuse or stash:
        fo = binding.forward(*args, gate=g, ckpt_every=ckpt_every, stash=stash)
        ckpt, z = fo["ckpt"], fo.get("z_stash")
    out = binding.backward(*args, d["dy"], gate=g, ckpt=ckpt, ckpt_every=ckpt_every, z_stash=z)
    st, detail = binding.sync_status(out["workspace"])
    assert st == binding.M2RNN_OK, (binding.status_string(st), detail)
    torch.cuda.synchronize()
    assert "df" not in out
    return {n: out[n].cpu().numpy() for n in ("dq", "dk", "dv", "da", "dalpha", "dbeta", "dW", "dw_r")}


@pytest.mark.parametrize("kernel_family", ["mma", "tcgen05", "simt"], indirect=True)
@pytest.mark.parametrize("B,N,T,K,V", [(2, 3, 37, 64, 64), (1, 2, 70, 32, 64)])
def test_gated_forward(kernel_family, B, N, T, K, V):
    inp, gs, ge = _gated_case(B, N, T, K, V, "bf16", seed=700 + T)
    got = _run_gated(inp, gs)
    y_ref, H_ref = oracle_forward(*_oracle_gated_args(inp, ge))
    assert max_abs(got["y"], y_ref) <= TOL_BF16_MAXABS_Y
    assert rel_fro(got["y"], y_ref) <= TOL_BF16_REL
    assert rel_fro(got["H_T"], H_ref) <= TOL_BF16_REL


@pytest.mark.parametrize("B,N,T,K,V,dtype,shared", [(1, 2, 45, 128, 128, "bf16", False),
                                                     (2, 4, 50, 64, 16, "bf16", True),
                                                     (1, 2, 20, 16, 16, "f32", False),
                                                     (1, 3, 9, 5, 7, "f32", False)])
def test_gated_forward_other_families(B, N, T, K, V, dtype, shared):
    inp, gs, ge = _gated_case(B, N, T, K, V, dtype, seed=710 + T, shared_qk=shared)
    got = _run_gated(inp, gs)
    y_ref, H_ref = oracle_forward(*_oracle_gated_args(inp, ge))
    if dtype == "f32":
        assert max_abs(got["y"], y_ref) <= TOL_F32 and rel_fro(got["H_T"], H_ref) <= TOL_F32
    else:
        assert max_abs(got["y"], y_ref) <= TOL_BF16_MAXABS_Y
        assert rel_fro(got["y"], y_ref) <= TOL_BF16_REL and rel_fro(got["H_T"], H_ref) <= TOL_BF16_REL


def _check_gated_grads(got, inp, ge, tol, label):
    ref = oracle_backward(*_oracle_gated_args(inp, ge), inp.exact["dy"])
    da, dal, dbe = gate_backward(ge["a"], ge["alpha"], ge["beta"], ref["df"])
    ref = dict(ref, da=da, dalpha=dal, dbeta=dbe)
    for name in ("dq", "dk", "dv", "da", "dalpha", "dbeta", "dW", "dw_r"):
        r = rel_fro(got[name], ref[name])
        assert r <= tol, (label, name, r)


@pytest.mark.parametrize("kernel_family", ["mma", "simt"], indirect=True)
@pytest.mark.parametrize("B,N,T,K,V,C,reuse", [(2, 2, 37, 64, 64, 14, False), (1, 3, 64, 32, 64, 18, True),
                                               (1, 1, 1, 64, 64, 14, False)])
def test_gated_backward(kernel_family, B, N, T, K, V, C, reuse):
    inp, gs, ge = _gated_case(B, N, T, K, V, "bf16", seed=720 + T)
    got = _run_gated(inp, gs, backward=True, ckpt_every=C, reuse=reuse)
    _check_gated_grads(got, inp, ge, TOL_BF16_REL, (kernel_family, B, N, T, K, V, C))


@pytest.mark.parametrize("B,N,T,K,V,dtype,shared,C", [(2, 4, 50, 64, 16, "bf16", True, 14),
                                                       (1, 2, 33, 128, 128, "bf16", False, 16),
                                                       (1, 2, 30, 16, 16, "f32", False, 8)])
def test_gated_backward_other_families(B, N, T, K, V, dtype, shared, C):
    inp, gs, ge = _gated_case(B, N, T, K, V, dtype, seed=730 + T, shared_qk=shared)
    got = _run_gated(inp, gs, backward=True, ckpt_every=C)
    _check_gated_grads(got, inp, ge, TOL_F32 if dtype == "f32" else TOL_BF16_REL, (B, N, T, K, V, dtype))


@pytest.mark.parametrize("B,N,T,K,V,C,shared", [(2, 2, 37, 64, 64, 14, False), (1, 3, 64, 32, 64, 18, False),
                                               (2, 4, 50, 64, 16, 28, True)])
def test_gated_backward_with_stash(B, N, T, K, V, C, shared):
    inp, gs, ge = _gated_case(B, N, T, K, V, "bf16", seed=760 + T, shared_qk=shared)
    got = _run_gated(inp, gs, backward=True, ckpt_every=C, stash=True)
    _check_gated_grads(got, inp, ge, TOL_BF16_REL, (B, N, T, K, V, C, "stash"))


def test_gated_backward_is_deterministic():
    inp, gs, _ = _gated_case(2, 4, 90, 64, 64, "bf16", seed=740)
    a = _run_gated(inp, gs, backward=True)
    b = _run_gated(inp, gs, backward=True)
    for name in a:
        assert np.array_equal(a[name], b[name]), name


def test_gated_full_size_properties():
    """The fwd+bwd workload's shape (B=4, heads=8, T=4096, K=V=64), run as
    the benchmark's gated block runs it (Z stash, 20-step chunks): dbeta is
    the (b, t)-sum of da, and dalpha the (b, t)-sum of da * s / (alpha
    sigmoid(a + beta)), recomputed from the kernel's own da in float64; and
    one head's gradients (dq, dk, dv, da, dalpha, dbeta) against the oracle."""
    inp, gs, ge = _gated_case(4, 8, 4096, 64, 64, "bf16", seed=750)
    got = _run_gated(inp, gs, backward=True, ckpt_every=20, stash=True)
    da = got["da"].astype(np.float64)
    assert np.all(np.isfinite(da))
    # fp32 sums of 16384 terms: bound the error by the sum of magnitudes
    assert np.all(np.abs(got["dbeta"] - da.sum(axis=(0, 1))) <= 1e-4 * np.abs(da).sum(axis=(0, 1)))
    x = ge["a"] + ge["beta"]
    s = np.logaddexp(0.0, x)
    sig = 0.5 * (1.0 + np.tanh(0.5 * x))
    terms = da * s / (ge["alpha"] * sig)
    assert np.all(np.abs(got["dalpha"] - terms.sum(axis=(0, 1))) <= 1e-4 * np.abs(terms).sum(axis=(0, 1)))
    n = 0
    e = inp.exact
    f = gate(ge["a"], ge["alpha"], ge["beta"])[:, :, n:n + 1]
    ref = oracle_backward(e["q"][:, :, n:n + 1], e["k"][:, :, n:n + 1], e["v"][:, :, n:n + 1], f, e["W"][n:n + 1],
                          e["w_r"][n:n + 1], e["dy"][:, :, n:n + 1])
    da_ref, dalpha_ref, dbeta_ref = gate_backward(ge["a"][:, :, n:n + 1], ge["alpha"][n:n + 1],
                                                  ge["beta"][n:n + 1], ref["df"])
    for name, r in (("dq", ref["dq"]), ("dk", ref["dk"]), ("dv", ref["dv"]), ("da", da_ref)):
        assert rel_fro(got[name][:, :, n:n + 1], r) <= TOL_BF16_REL, (name, rel_fro(got[name][:, :, n:n + 1], r))
    # The head's gate-parameter gradients (sums over every b and t) against the oracle's.
    for name, r in (("dalpha", dalpha_ref), ("dbeta", dbeta_ref)):
        assert rel_fro(got[name][n:n + 1], r) <= TOL_BF16_REL, (name, rel_fro(got[name][n:n + 1], r))


# ---------------------------------------------------------------------------
# Output path
# ---------------------------------------------------------------------------

def _run_norm(store, eps, backward=False):
    import torch
    from matrix_state_non_gb300 import binding
    d = {n: _dev(x) for n, x in store.items()}
    if not backward:
        out, rstd = binding.output_norm(d["y"], d["g"], d["w"], eps=eps, want_rstd=True)
        torch.cuda.synchronize()
        return out.cpu().numpy(), rstd.cpu().numpy()
    res = binding.output_norm_backward(d["y"], d["g"], d["w"], d["dout"], eps=eps)
    torch.cuda.synchronize()
    return {n: v.cpu().numpy() for n, v in res.items()}


# widths d = N V: 512 (a warp per row, 4 groups of 4 per lane), 256 (the
# pages' 16 heads x 16), 15 (not a multiple of 4: scalar path), 960 (a warp
# per row, 8 groups per lane, ragged), 1600 (a block per row, 256 threads x
# 2 groups), 4100 (256 threads x 5 of 8 groups, ragged), 16384 (the widest,
# N = V = 128, 512 threads), 4 (one head, one group).
NORM_SHAPES = [(2, 33, 8, 64), (1, 17, 16, 16), (2, 5, 3, 5), (1, 9, 12, 80), (2, 7, 16, 100),
               (1, 3, 41, 100), (1, 2, 128, 128), (1, 1, 1, 4)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,N,V", NORM_SHAPES)
def test_output_norm(dtype, B, T, N, V):
    store, exact = make_norm_inputs(B, T, N, V, dtype, seed=800 + N * V)
    eps = 1e-6
    out, rstd = _run_norm(store, eps)
    ref = output_norm(exact["y"], exact["g"], exact["w"], eps)
    assert rel_fro(out, ref) <= 1e-5 and max_abs(out, ref) <= 1e-4 * max(1.0, np.abs(ref).max())
    x = exact["y"] * exact["g"]
    s_ref = (np.sum(x * x, axis=(2, 3)) / (N * V) + eps) ** -0.5
    np.testing.assert_allclose(rstd, s_ref, rtol=1e-5)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,N,V", NORM_SHAPES)
def test_output_norm_backward(dtype, B, T, N, V):
    store, exact = make_norm_inputs(B, T, N, V, dtype, seed=900 + N * V)
    eps = 1e-6
    got = _run_norm(store, eps, backward=True)
    dy, dg, dw = output_norm_backward(exact["y"], exact["g"], exact["w"], exact["dout"], eps)
    for name, ref in (("dy", dy), ("dg", dg), ("dw", dw)):
        assert rel_fro(got[name], ref) <= 1e-5, (name, rel_fro(got[name], ref))


def test_output_norm_zero_eps_and_determinism():
    store, exact = make_norm_inputs(3, 40, 8, 64, "bf16", seed=950)
    out, _ = _run_norm(store, 0.0)
    assert rel_fro(out, output_norm(exact["y"], exact["g"], exact["w"], 0.0)) <= 1e-5
    a = _run_norm(store, 1e-5, backward=True)
    b = _run_norm(store, 1e-5, backward=True)
    for name in a:
        assert np.array_equal(a[name], b[name]), name


def test_output_norm_full_size():
    """The fwd+bwd workload's output width and token count (B=4, T=4096,
    heads=8, V=64), every element against the oracle."""
    store, exact = make_norm_inputs(4, 4096, 8, 64, "bf16", seed=960)
    out, _ = _run_norm(store, 1e-6)
    assert rel_fro(out, output_norm(exact["y"], exact["g"], exact["w"], 1e-6)) <= 1e-5
    got = _run_norm(store, 1e-6, backward=True)
    dy, dg, dw = output_norm_backward(exact["y"], exact["g"], exact["w"], exact["dout"], 1e-6)
    for name, ref in (("dy", dy), ("dg", dg), ("dw", dw)):
        assert rel_fro(got[name], ref) <= 1e-5, (name, rel_fro(got[name], ref))
