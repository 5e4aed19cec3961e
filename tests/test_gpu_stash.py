"""GPU parity for the backward that reads the forward's Z stash (V = 64
warp-MMA kernels): the forward leaves Z_t of every step in fp16, and the
backward advances the state from each checkpoint by the gate blend alone
instead of rerunning the transform and tanh (Eq. 10-11 of the reading notes,
section 2.1; the backward of section 2.7).

Every case is compared with the float64 oracle at the bf16 tolerances; the
forward's own outputs must not change when it writes the stash.
"""
import numpy as np
import pytest

from matrix_state_non_gb300.inputs import WORKLOADS, make_gate_inputs, make_inputs, make_workload
from oracle import backward as oracle_backward
from oracle import gate, gate_backward
from parity_util import IN_NAMES, TOL_BF16_REL, check_grads, gpu_backward, oracle_args, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,N,T,K,V,C", [(2, 3, 37, 64, 64, 14), (1, 2, 100, 32, 64, 14), (1, 1, 1, 64, 64, 14),
                                         (1, 2, 64, 128, 64, 18), (2, 2, 45, 64, 64, 5), (1, 1, 14, 64, 64, 14),
                                         (1, 1, 15, 16, 64, 14), (1, 2, 57, 64, 64, 17)])
def test_stash_backward_matches_oracle(B, N, T, K, V, C):
    inp = make_inputs(B, N, T, K, V, "bf16", seed=600 + T + C, with_dy=True)
    dH = np.random.default_rng(T).standard_normal((B, N, K, V)).astype(np.float32)
    got = gpu_backward(inp, dH_T=dH, ckpt_every=C, stash=True)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], dH.astype(np.float64))
    check_grads(got, ref, "bf16", label=(B, N, T, K, V, C))


def test_stash_with_initial_state_and_clipping():
    B, N, T, K, V = 2, 2, 60, 64, 64
    inp = make_inputs(B, N, T, K, V, "bf16", seed=611, with_dy=True)
    H0 = np.random.default_rng(3).uniform(-0.9, 0.9, (B, N, K, V)).astype(np.float32)
    got = gpu_backward(inp, ckpt_every=14, stash=True, H_0=H0, want_dH0=True)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], None, H_0=H0.astype(np.float64))
    check_grads(got, ref, "bf16", label="H_0")
    got = gpu_backward(inp, ckpt_every=14, stash=True, state_grad_clip=0.05)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], None, state_grad_clip=0.05)
    check_grads(got, ref, "bf16", label="clip")


def test_stash_shared_qk_and_gate():
    import torch
    from matrix_state_non_gb300 import binding
    B, N, T, K, V = 2, 4, 50, 64, 64
    inp = make_inputs(B, N, T, K, V, "bf16", seed=612, with_dy=True)
    for name in ("q", "k"):
        inp.store[name] = np.ascontiguousarray(inp.store[name][:, :, :1])
        inp.exact[name] = np.ascontiguousarray(inp.exact[name][:, :, :1])
    gs, ge = make_gate_inputs(B, T, N, "bf16", seed=613)
    d = binding.to_device(inp)

    class _S:
        store = gs
    g = binding.to_device(_S)
    gt = (g["a"], g["alpha"], g["beta"])
    args = (d["q"], d["k"], d["v"], None, d["W"], d["w_r"])
    fo = binding.forward(*args, gate=gt, ckpt_every=14, stash=True)
    out = binding.backward(*args, d["dy"], gate=gt, ckpt=fo["ckpt"], ckpt_every=14, z_stash=fo["z_stash"])
    st, detail = binding.sync_status(out["workspace"])
    assert st == binding.M2RNN_OK, (binding.status_string(st), detail)
    torch.cuda.synchronize()
    e = inp.exact
    f = gate(ge["a"], ge["alpha"], ge["beta"])
    ref = oracle_backward(e["q"], e["k"], e["v"], f, e["W"], e["w_r"], e["dy"])
    da, dal, dbe = gate_backward(ge["a"], ge["alpha"], ge["beta"], ref["df"])
    ref = dict(ref, da=da, dalpha=dal, dbeta=dbe)
    for name in ("dq", "dk", "dv", "da", "dalpha", "dbeta", "dW", "dw_r"):
        r = rel_fro(out[name].cpu().numpy(), ref[name])
        assert r <= TOL_BF16_REL, (name, r)


def test_forward_outputs_unchanged_by_the_stash():
    """The stash leaves the outputs of the kernel that writes it (the
    warp-MMA forward at V = 64) unchanged."""
    import torch
    from matrix_state_non_gb300 import binding
    inp = make_inputs(2, 2, 90, 64, 64, "bf16", seed=614)
    d = binding.to_device(inp)
    assert binding.m2rnn_path(64, 64, binding.M2RNN_BF16) == 2  # the same kernel with and without the stash
    a = binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=14)
    b = binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=14, stash=True)
    torch.cuda.synchronize()
    for name in ("y", "H_T", "ckpt"):
        assert torch.equal(a[name], b[name]), name
    # The stash holds fp16(Z_t): every value inside [-1, 1].
    z = b["z_stash"].view(torch.float16).float()
    assert z.numel() == 2 * 90 * 2 * 64 * 64 and bool((z.abs() <= 1.0).all())


def test_stash_backward_is_deterministic():
    inp = make_inputs(2, 2, 80, 64, 64, "bf16", seed=615, with_dy=True)
    a = gpu_backward(inp, ckpt_every=18, stash=True)
    b = gpu_backward(inp, ckpt_every=18, stash=True)
    for name in a:
        assert np.array_equal(a[name], b[name]), name


def test_stash_backward_full_size_sampled_head():
    """The forward+backward workload as the benchmark runs it (stash and
    checkpoints from the forward): one head's gradients over every batch
    element against the oracle."""
    name = "fwdbwd_bf16_k64"
    w = WORKLOADS[name]
    inp = make_workload(name)
    got = gpu_backward(inp, ckpt_every=20, stash=True)  # the benchmark's chunk length
    n = 0
    ref = oracle_backward(*oracle_args(inp, slice(None), slice(n, n + 1)), inp.exact["dy"][:, :, n:n + 1])
    sub = {"dq": got["dq"][:, :, n:n + 1], "dk": got["dk"][:, :, n:n + 1], "dv": got["dv"][:, :, n:n + 1],
           "df": got["df"][:, :, n:n + 1], "dW": got["dW"][n:n + 1], "dw_r": got["dw_r"][n:n + 1]}
    check_grads(sub, ref, "bf16", label=name)
    assert w["V"] == 64


# V = 16 (the multi-value heads of the reading notes, section 2.4): the stash
# is written by the register-resident V = 16 forward and read by its backward.
@pytest.mark.parametrize("B,N,T,K,C,shared", [(2, 4, 50, 64, 14, True), (1, 3, 100, 64, 28, False),
                                             (2, 2, 33, 128, 16, True), (1, 2, 1, 32, 14, False),
                                             (1, 2, 64, 16, 32, True), (2, 3, 81, 64, 20, True),
                                             (1, 2, 47, 128, 10, False), (1, 2, 39, 80, 9, True)])
def test_stash_backward_v16_matches_oracle(B, N, T, K, C, shared):
    inp = make_inputs(B, N, T, K, 16, "bf16", seed=620 + T + C, with_dy=True)
    if shared:
        for name in ("q", "k"):
            inp.store[name] = np.ascontiguousarray(inp.store[name][:, :, :1])
            inp.exact[name] = np.ascontiguousarray(inp.exact[name][:, :, :1])
    H0 = np.random.default_rng(T).uniform(-0.9, 0.9, (B, N, K, 16)).astype(np.float32)
    got = gpu_backward(inp, ckpt_every=C, stash=True, H_0=H0, want_dH0=True)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], None, H_0=H0.astype(np.float64))
    check_grads(got, ref, "bf16", label=(B, N, T, K, C, shared))


def test_stash_v16_clipping_and_full_size():
    """Clipped state gradients with the stash, then the V = 16 forward+backward
    workload (B=4, 16 heads, T=4096, K=64, shared q/k) as the benchmark runs
    it, one head against the oracle."""
    inp = make_inputs(1, 2, 60, 64, 16, "bf16", seed=630, with_dy=True)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], None, state_grad_clip=0.05)
    for C in (28, 14):  # the single-warp and the pipelined kernel
        got = gpu_backward(inp, ckpt_every=C, stash=True, state_grad_clip=0.05)
        check_grads(got, ref, "bf16", label=("clip", C))
    name = "mv_bf16_k64v16"
    inp = make_workload(name)
    got = gpu_backward(inp, ckpt_every=20, stash=True)  # the benchmark's chunk length for V = 16
    e = inp.exact
    n = WORKLOADS[name]["N"] - 1
    ref = oracle_backward(e["q"], e["k"], e["v"][:, :, n:n + 1], e["f"][:, :, n:n + 1], e["W"][n:n + 1],
                          e["w_r"][n:n + 1], e["dy"][:, :, n:n + 1])
    # q, k are shared: their gradients sum over every head, so compare the
    # per-head outputs of head n only.
    sub = {"dv": got["dv"][:, :, n:n + 1], "df": got["df"][:, :, n:n + 1], "dW": got["dW"][n:n + 1],
           "dw_r": got["dw_r"][n:n + 1]}
    for k_, v_ in sub.items():
        assert rel_fro(v_, ref[k_]) <= TOL_BF16_REL, (k_, rel_fro(v_, ref[k_]))
