"""GPU parity for multi-value heads: one q/k shared by every value head
(section 2.4 of the M2RNN reading notes; the paper's configuration uses
K = 64, V = 16), with dq, dk summed over the heads (section 2.7).  Every
kernel family against the float64 oracle."""
import copy

import numpy as np
import pytest

from matrix_state_non_gb300.inputs import make_inputs
from oracle import backward as oracle_backward
from oracle import forward as oracle_forward
from parity_util import check_forward, check_grads, gpu_backward, gpu_forward, oracle_args

pytestmark = pytest.mark.gpu


def shared_inputs(B, N, T, K, V, dtype, seed, with_dy=False):
    """Seeded inputs with q, k reduced to one head ([B,T,1,K])."""
    inp = make_inputs(B, N, T, K, V, dtype, seed=seed, with_dy=with_dy)
    out = copy.copy(inp)
    out.store = dict(inp.store)
    out.exact = dict(inp.exact)
    for name in ("q", "k"):
        out.store[name] = np.ascontiguousarray(inp.store[name][:, :, :1])
        out.exact[name] = np.ascontiguousarray(inp.exact[name][:, :, :1])
    return out


@pytest.mark.parametrize("kernel_family", ["mma", "tcgen05", "simt"], indirect=True)
@pytest.mark.parametrize("B,N,T,K,V", [(2, 4, 37, 64, 64), (1, 3, 50, 32, 64)])
def test_forward_shared_qk(kernel_family, B, N, T, K, V):
    inp = shared_inputs(B, N, T, K, V, "bf16", seed=400 + T)
    got = gpu_forward(inp, ckpt_every=16)
    y_ref, H_ref = oracle_forward(*oracle_args(inp))
    check_forward(got, y_ref, H_ref, "bf16", label=(kernel_family, B, N, T, K, V))


@pytest.mark.parametrize("B,N,T,K,V,dtype", [(2, 8, 40, 64, 16, "bf16"), (1, 4, 30, 64, 16, "f32"),
                                             (1, 2, 33, 128, 128, "bf16")])
def test_forward_shared_qk_other_shapes(B, N, T, K, V, dtype):
    """The paper's multi-value shape (K = 64, V = 16) and the wide heads."""
    inp = shared_inputs(B, N, T, K, V, dtype, seed=410 + T)
    got = gpu_forward(inp)
    y_ref, H_ref = oracle_forward(*oracle_args(inp))
    check_forward(got, y_ref, H_ref, dtype, label=(B, N, T, K, V, dtype))


@pytest.mark.parametrize("kernel_family", ["mma", "simt"], indirect=True)
@pytest.mark.parametrize("B,N,T,K,V,C", [(2, 4, 37, 64, 64, 14), (1, 3, 45, 32, 64, 18)])
def test_backward_shared_qk(kernel_family, B, N, T, K, V, C):
    inp = shared_inputs(B, N, T, K, V, "bf16", seed=420 + T, with_dy=True)
    dH = np.random.default_rng(6).standard_normal((B, N, K, V)).astype(np.float32)
    got = gpu_backward(inp, dH_T=dH, ckpt_every=C, use_fwd_ckpt=True)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], dH.astype(np.float64))
    assert got["dq"].shape == (B, T, 1, K) and got["dk"].shape == (B, T, 1, K)
    check_grads(got, ref, "bf16", label=(kernel_family, B, N, T, K, V, C))


@pytest.mark.parametrize("B,N,T,K,V,dtype", [(2, 8, 40, 64, 16, "bf16"), (1, 4, 30, 64, 16, "f32")])
def test_backward_shared_qk_paper_shape(B, N, T, K, V, dtype):
    inp = shared_inputs(B, N, T, K, V, dtype, seed=430 + T, with_dy=True)
    got = gpu_backward(inp, ckpt_every=8)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"])
    check_grads(got, ref, dtype, label=(B, N, T, K, V, dtype))


@pytest.mark.parametrize("kernel_family", ["auto", "mma"], indirect=True)
def test_decode_shared_qk(kernel_family):
    import torch
    from matrix_state_non_gb300 import binding
    B, N, T, K, V = 2, 4, 10, 64, 64
    inp = shared_inputs(B, N, T, K, V, "bf16", seed=440)
    d = binding.to_device(inp)
    H = torch.zeros((B, N, K, V), device="cuda", dtype=torch.float32)
    ys = []
    for t in range(T):
        step = [d[n][:, t].contiguous() for n in ("q", "k", "v", "f")]
        ys.append(binding.decode_step(H, *step, d["W"], d["w_r"]).cpu().numpy())
    torch.cuda.synchronize()
    y_ref, H_ref = oracle_forward(*oracle_args(inp))
    check_forward({"y": np.stack(ys, axis=1), "H_T": H.cpu().numpy()}, y_ref, H_ref, "bf16")


@pytest.mark.parametrize("shared", [True, False])
@pytest.mark.parametrize("B,N,T,K", [(2, 4, 77, 64), (1, 3, 33, 16), (1, 2, 40, 128), (1, 1, 1, 64)])
def test_forward_v16_register_kernel(shared, B, N, T, K):
    """The V = 16 register-resident kernel (bf16): y, H_T and checkpoints
    from a non-zero initial state, several tiles and a ragged last tile."""
    V = 16
    maker = shared_inputs if shared else (lambda *a, **kw: make_inputs(*a, **kw))
    inp = maker(B, N, T, K, V, "bf16", seed=450 + T + K)
    H0 = np.random.default_rng(T).uniform(-0.9, 0.9, (B, N, K, V)).astype(np.float32)
    got = gpu_forward(inp, ckpt_every=8, H_0=H0)
    y_ref, H_ref, Hs, _ = oracle_forward(*oracle_args(inp), return_states=True, H_0=H0.astype(np.float64))
    check_forward(got, y_ref, H_ref, "bf16", label=(shared, B, N, T, K))
    from parity_util import rel_fro
    for c in range((T - 1) // 8):
        assert rel_fro(got["ckpt"][:, :, c], Hs[(c + 1) * 8]) <= 1e-2


@pytest.mark.parametrize("shared", [True, False])
@pytest.mark.parametrize("B,N,T,K,C", [(2, 4, 45, 64, 8), (1, 3, 70, 16, 32), (1, 2, 33, 128, 16),
                                       (1, 2, 5, 64, 1), (2, 2, 64, 32, 13), (2, 2, 61, 64, 20),
                                       (1, 2, 50, 48, 20), (1, 2, 40, 128, 10), (1, 2, 57, 96, 7),
                                       (1, 2, 90, 64, 25)])
def test_backward_v16_register_kernel(shared, B, N, T, K, C):
    """The V = 16 register-resident backward (bf16): every gradient and dH_0
    from a non-zero initial state, several chunks and a ragged first chunk.
    Chunks of up to 20 steps (10 with K > 64) run the pipelined kernel
    (rebuild and chain warps per row block), longer ones the single-warp
    kernel: both are covered."""
    V = 16
    maker = shared_inputs if shared else (lambda *a, **kw: make_inputs(*a, **kw))
    inp = maker(B, N, T, K, V, "bf16", seed=460 + T + K + C, with_dy=True)
    rng = np.random.default_rng(C)
    H0 = rng.uniform(-0.9, 0.9, (B, N, K, V)).astype(np.float32)
    dH = rng.standard_normal((B, N, K, V)).astype(np.float32)
    got = gpu_backward(inp, dH_T=dH, ckpt_every=C, use_fwd_ckpt=(C % 2 == 0), H_0=H0, want_dH0=True)
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], dH.astype(np.float64), H_0=H0.astype(np.float64))
    check_grads(got, ref, "bf16", label=(shared, B, N, T, K, C))


def test_forward_v16_full_size_sampled_heads():
    """The V = 16 forward at the benchmark's size (B=4, 16 heads, T=4096,
    K=64, one q/k shared by the heads; the pipelined compute/readout kernel):
    y and H_T of sampled heads against the oracle."""
    from matrix_state_non_gb300.inputs import WORKLOADS, make_workload
    name = "mv_bf16_k64v16"
    w = WORKLOADS[name]
    inp = make_workload(name)
    got = gpu_forward(inp, ckpt_every=20)
    e = inp.exact
    for b, n in [(0, 0), (w["B"] - 1, w["N"] - 1), (1, 7)]:
        y_ref, H_ref = oracle_forward(e["q"][b:b + 1], e["k"][b:b + 1], e["v"][b:b + 1, :, n:n + 1],
                                      e["f"][b:b + 1, :, n:n + 1], e["W"][n:n + 1], e["w_r"][n:n + 1])
        sub = {"y": got["y"][b:b + 1, :, n:n + 1], "H_T": got["H_T"][b:b + 1, n:n + 1]}
        check_forward(sub, y_ref, H_ref, "bf16", label=(name, b, n))
