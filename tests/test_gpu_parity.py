"""GPU parity: the CUDA path (called through the C ABI) against the float64
oracle on the same seeded inputs.

Tolerances (stated for the M2RNN scans): bf16 inputs with fp32 state need
max-abs <= 3e-2 on y and relative Frobenius <= 1e-2 on y, H_T and every
gradient; all-fp32 runs need <= 1e-4.  Small cases run the oracle on every
chain; the full-size workloads run the GPU on the whole batch in the same
launch configuration the benchmark uses and compare sampled chains.
"""
import numpy as np
import pytest

from matrix_state_non_gb300.inputs import WORKLOADS, from_exact, make_inputs, make_workload
from oracle import backward as oracle_backward
from oracle import forward as oracle_forward
from parity_util import (check_forward, check_grads, gpu_backward, gpu_forward, max_abs,
                         oracle_args, rel_fro)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from matrix_state_non_gb300 import binding
    binding.load()


# ---------------------------------------------------------------------------
# Forward, small shapes: every chain against the oracle
# ---------------------------------------------------------------------------
SMALL_FWD = [
    # (B, N, T, K, V, dtype)
    (1, 2, 64, 16, 16, "f32"),
    (1, 1, 1, 64, 64, "bf16"),
    (1, 1, 2, 64, 64, "bf16"),
    (2, 3, 37, 64, 64, "bf16"),
    (1, 2, 70, 16, 64, "bf16"),
    (1, 1, 97, 128, 64, "bf16"),
    (2, 1, 33, 48, 64, "bf16"),
    (2, 2, 45, 128, 128, "bf16"),
    (1, 2, 40, 64, 128, "bf16"),
    (1, 1, 20, 32, 128, "bf16"),
    (2, 2, 19, 32, 32, "bf16"),
    (1, 3, 25, 7, 5, "f32"),
    (1, 2, 33, 100, 48, "bf16"),
]


@pytest.mark.parametrize("B,N,T,K,V,dtype", SMALL_FWD)
def test_forward_small_matches_oracle(B, N, T, K, V, dtype):
    inp = make_inputs(B, N, T, K, V, dtype, seed=B * 1000 + T + K + V)
    got = gpu_forward(inp)
    y_ref, H_ref = oracle_forward(*oracle_args(inp))
    check_forward(got, y_ref, H_ref, dtype, label=(B, N, T, K, V, dtype))


def test_tiny_f32_workload():
    inp = make_workload("tiny_f32")
    got = gpu_forward(inp)
    y_ref, H_ref = oracle_forward(*oracle_args(inp))
    check_forward(got, y_ref, H_ref, "f32")


@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (16, 16)])
def test_forget_one_keeps_zero_state_on_gpu(K, V):
    """f = 1: the state stays exactly 0 and y = w_r * v (bf16 product, fp32 out)."""
    inp = make_inputs(2, 2, 40, K, V, "bf16", seed=5, f_mode="ones")
    got = gpu_forward(inp)
    assert np.all(got["H_T"] == 0.0)
    ref = inp.exact["w_r"][None, None] * inp.exact["v"]
    assert max_abs(got["y"], ref) <= 1e-6


@pytest.mark.parametrize("K,V", [(64, 64), (128, 128)])
def test_memoryless_case_on_gpu(K, V):
    """f = 0, W = 0: H_t = tanh(k_t v_t^T) at every step."""
    inp = make_inputs(1, 2, 9, K, V, "bf16", seed=6, f_mode="zeros")
    ex = dict(inp.exact)
    ex["W"] = np.zeros_like(ex["W"])
    inp = from_exact(ex, "bf16")
    got = gpu_forward(inp)
    H_ref = np.tanh(ex["k"][:, -1, :, :, None] * ex["v"][:, -1, :, None, :])
    assert max_abs(got["H_T"], H_ref) <= 2e-3
    y_ref, _ = oracle_forward(*oracle_args(inp))
    check_forward(got, y_ref, H_ref, "bf16")


@pytest.mark.parametrize("K,V", [(64, 64), (128, 128)])
def test_identity_transition_on_gpu(K, V):
    """W = I (the paper's initialisation)."""
    inp = make_inputs(2, 2, 50, K, V, "bf16", seed=7)
    ex = dict(inp.exact)
    ex["W"] = np.broadcast_to(np.eye(V), ex["W"].shape).copy()
    inp = from_exact(ex, "bf16")
    got = gpu_forward(inp)
    y_ref, H_ref = oracle_forward(*oracle_args(inp))
    check_forward(got, y_ref, H_ref, "bf16")


def test_theorem1_case_on_gpu():
    """f = 0, w_r = 0, q = k = e_1: only row 1 is non-zero (a tanh RNN)."""
    B, N, T, K, V = 1, 2, 40, 64, 64
    inp = make_inputs(B, N, T, K, V, "bf16", seed=8, f_mode="zeros")
    ex = dict(inp.exact)
    e1 = np.zeros(K)
    e1[0] = 1.0
    ex["q"] = np.broadcast_to(e1, ex["q"].shape).copy()
    ex["k"] = ex["q"].copy()
    ex["w_r"] = np.zeros_like(ex["w_r"])
    inp = from_exact(ex, "bf16")
    got = gpu_forward(inp)
    assert np.all(got["H_T"][:, :, 1:, :] == 0.0)
    y_ref, H_ref = oracle_forward(*oracle_args(inp))
    check_forward(got, y_ref, H_ref, "bf16")


@pytest.mark.parametrize("K,V,C", [(64, 64, 16), (128, 128, 32), (16, 16, 8)])
def test_checkpoints_match_oracle_states(K, V, C):
    inp = make_inputs(1, 2, 70, K, V, "bf16", seed=9)
    got = gpu_forward(inp, ckpt_every=C)
    _, _, Hs, _ = oracle_forward(*oracle_args(inp), return_states=True)
    nck = (70 - 1) // C
    assert got["ckpt"].shape == (1, 2, nck, K, V)
    for c in range(nck):
        ref = Hs[(c + 1) * C]  # [B,N,K,V]
        assert rel_fro(got["ckpt"][:, :, c], ref) <= 1e-2


def test_forward_is_deterministic():
    inp = make_inputs(2, 4, 100, 64, 64, "bf16", seed=10)
    a = gpu_forward(inp)
    b = gpu_forward(inp)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["H_T"], b["H_T"])


# ---------------------------------------------------------------------------
# Forward, full-size workloads: whole batch on the GPU, sampled chains checked
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["fwd_bf16_k64", "fwd_bf16_k128", "fwd_bf16_16k"])
def test_forward_full_size_sampled_chains(name):
    w = WORKLOADS[name]
    inp = make_workload(name)
    got = gpu_forward(inp)
    rng = np.random.default_rng(123)
    samples = [(0, 0), (w["B"] - 1, w["N"] - 1), (int(rng.integers(w["B"])), int(rng.integers(w["N"])))]
    for b, n in samples:
        y_ref, H_ref = oracle_forward(*oracle_args(inp, slice(b, b + 1), slice(n, n + 1)))
        sub = {"y": got["y"][b:b + 1, :, n:n + 1], "H_T": got["H_T"][b:b + 1, n:n + 1]}
        check_forward(sub, y_ref, H_ref, "bf16", label=(name, b, n))


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------
SMALL_BWD = [
    # (B, N, T, K, V, dtype, ckpt_every, with dH_T, reuse forward checkpoints)
    (1, 2, 64, 16, 16, "f32", 16, True, False),
    (1, 1, 1, 64, 64, "bf16", 16, True, False),
    (2, 2, 37, 64, 64, "bf16", 16, False, False),
    (2, 2, 70, 64, 64, "bf16", 18, True, True),
    (1, 2, 45, 128, 128, "bf16", 16, True, False),
    (2, 1, 33, 32, 64, "bf16", 8, True, True),
    (1, 3, 25, 7, 5, "f32", 4, True, False),
]


@pytest.mark.parametrize("B,N,T,K,V,dtype,C,with_dH,reuse", SMALL_BWD)
def test_backward_small_matches_oracle(B, N, T, K, V, dtype, C, with_dH, reuse):
    inp = make_inputs(B, N, T, K, V, dtype, seed=77 + T, with_dy=True)
    dH = np.random.default_rng(3).standard_normal((B, N, K, V)).astype(np.float32) if with_dH else None
    got = gpu_backward(inp, dH_T=dH, ckpt_every=C, use_fwd_ckpt=reuse)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"],
                          None if dH is None else dH.astype(np.float64))
    check_grads(got, ref, dtype, label=(B, N, T, K, V, dtype, C))


@pytest.mark.parametrize("n", [0, 7])
def test_backward_full_size_sampled_head(n):
    """Forward+backward workload: the whole batch on the GPU (checkpoints from
    the forward, as the benchmark runs it); one head's gradients over every
    batch element against the oracle (dW and dw_r sum over b).  Head 0's
    state gradient grows ~9x over the 4096 steps back, which amplifies any
    error in the forward's Z_t: the case that needs the hi/lo state operand."""
    name = "fwdbwd_bf16_k64"
    w = WORKLOADS[name]
    assert n < w["N"]
    inp = make_workload(name)
    got = gpu_backward(inp, ckpt_every=20, use_fwd_ckpt=True)  # the benchmark's chunk length
    ref = oracle_backward(*oracle_args(inp, slice(None), slice(n, n + 1)),
                          inp.exact["dy"][:, :, n:n + 1])
    sub = {"dq": got["dq"][:, :, n:n + 1], "dk": got["dk"][:, :, n:n + 1],
           "dv": got["dv"][:, :, n:n + 1], "df": got["df"][:, :, n:n + 1],
           "dW": got["dW"][n:n + 1], "dw_r": got["dw_r"][n:n + 1]}
    check_grads(sub, ref, "bf16", label=(name, n))


@pytest.mark.parametrize("B,N,T,K,V,C,reuse,with_dH", [
    (2, 3, 50, 128, 128, 40, True, True),    # chunks longer than the 16 staged steps, ragged last chunk
    (1, 2, 37, 16, 128, 7, False, True),     # one compute warp beside the idle warps of the dW read-back
    (1, 1, 33, 96, 128, 16, True, False),    # six compute warps, no dH_T
    (1, 1, 5, 64, 128, 1, False, True),      # one-step chunks
    (1, 2, 1, 128, 128, 16, False, True),    # a single step
    (8, 16, 24, 128, 128, 16, True, True),   # the wide-head workload's grid (B=8, 16 heads), short T
    (2, 2, 45, 128, 128, 8, True, True),     # K = 128, C <= 16: the all-tcgen05 kernel, ragged last chunk
    (1, 3, 17, 128, 128, 1, True, True),     # one-step chunks (every step a rerun and a walk)
    (2, 1, 64, 128, 128, 12, False, True),   # checkpoints recomputed by the caller layer, 12-step chunks
    (1, 2, 96, 128, 128, 16, True, False),   # the longest chunks, no dH_T
])
def test_backward_v128_tensor_core(B, N, T, K, V, C, reuse, with_dH):
    """The V = 128 backward against the oracle: K = 128 with chunks of at
    most 16 steps runs every product on tcgen05; other K, or longer chunks,
    run the warp-MMA chain with the tcgen05 dW (it takes every K % 16 == 0;
    the forward that writes the checkpoints is the tcgen05 kernel for K =
    32, 64, 128 and the SIMT kernel otherwise)."""
    inp = make_inputs(B, N, T, K, V, "bf16", seed=500 + T + K, with_dy=True)
    dH = np.random.default_rng(9).standard_normal((B, N, K, V)).astype(np.float32) if with_dH else None
    got = gpu_backward(inp, dH_T=dH, ckpt_every=C, use_fwd_ckpt=reuse)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], None if dH is None else dH.astype(np.float64))
    check_grads(got, ref, "bf16", label=(B, N, T, K, V, C))


def test_backward_v128_full_size_sampled_head():
    """The wide-head training workload as the benchmark runs it (B=8, 16
    heads, T=1024, K=V=128: tcgen05 forward writing checkpoints every 8
    steps, then the all-tcgen05 V = 128 backward): one head's gradients over
    every batch element against the oracle."""
    name = "fwdbwd_bf16_k128"
    inp = make_workload(name)
    n = 5
    got = gpu_backward(inp, ckpt_every=8, use_fwd_ckpt=True)
    ref = oracle_backward(*oracle_args(inp, slice(None), slice(n, n + 1)),
                          inp.exact["dy"][:, :, n:n + 1])
    sub = {"dq": got["dq"][:, :, n:n + 1], "dk": got["dk"][:, :, n:n + 1],
           "dv": got["dv"][:, :, n:n + 1], "df": got["df"][:, :, n:n + 1],
           "dW": got["dW"][n:n + 1], "dw_r": got["dw_r"][n:n + 1]}
    check_grads(sub, ref, "bf16", label=(name, n))


def test_backward_is_deterministic():
    for V in (64, 128):
        inp = make_inputs(2, 2, 80, 64, V, "bf16", seed=12, with_dy=True)
        a = gpu_backward(inp, ckpt_every=16)
        b = gpu_backward(inp, ckpt_every=16)
        for name in a:
            assert np.array_equal(a[name], b[name]), (V, name)


# ---------------------------------------------------------------------------
# Every kernel family on the shapes they share (V = 64): the dispatcher picks
# the warp-MMA forward (the tcgen05 one where the Z stash is written);
# M2RNN_KERNEL selects each family explicitly.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("kernel_family", ["mma", "tcgen05", "simt"], indirect=True)
@pytest.mark.parametrize("B,N,T,K,V", [(2, 3, 37, 64, 64), (1, 2, 70, 16, 64), (1, 1, 97, 128, 64),
                                       (2, 1, 33, 48, 64), (1, 1, 1, 64, 64)])
def test_forward_each_kernel_family(kernel_family, B, N, T, K, V):
    from matrix_state_non_gb300 import binding
    expect = {"mma": 2, "tcgen05": 1, "simt": 0}[kernel_family]
    assert binding.m2rnn_path(K, V, binding.M2RNN_BF16) == expect
    inp = make_inputs(B, N, T, K, V, "bf16", seed=T + K)
    got = gpu_forward(inp, ckpt_every=16)
    y_ref, H_ref, Hs, _ = oracle_forward(*oracle_args(inp), return_states=True)
    check_forward(got, y_ref, H_ref, "bf16", label=(kernel_family, B, N, T, K, V))
    for c in range((T - 1) // 16):
        assert rel_fro(got["ckpt"][:, :, c], Hs[(c + 1) * 16]) <= 1e-2


@pytest.mark.parametrize("kernel_family", ["mma", "simt"], indirect=True)
@pytest.mark.parametrize("B,N,T,K,V,C", [(2, 2, 37, 64, 64, 16), (1, 1, 70, 32, 64, 32),
                                         (1, 2, 129, 16, 64, 7), (1, 1, 5, 64, 64, 1),
                                         (1, 1, 64, 128, 64, 28), (1, 1, 200, 64, 64, 14),
                                         (2, 1, 90, 32, 64, 15), (1, 2, 100, 64, 64, 16)])
def test_backward_each_kernel_family(kernel_family, B, N, T, K, V, C):
    inp = make_inputs(B, N, T, K, V, "bf16", seed=T + C, with_dy=True)
    dH = np.random.default_rng(4).standard_normal((B, N, K, V)).astype(np.float32)
    got = gpu_backward(inp, dH_T=dH, ckpt_every=C)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], dH.astype(np.float64))
    check_grads(got, ref, "bf16", label=(kernel_family, B, N, T, K, V, C))


def test_backward_long_chunk_falls_back():
    """Chunks longer than the warp-MMA backward's chunk limit (20
    steps) run on the CUDA cores."""
    inp = make_inputs(1, 1, 300, 64, 64, "bf16", seed=21, with_dy=True)
    got = gpu_backward(inp, ckpt_every=64)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"])
    check_grads(got, ref, "bf16")
