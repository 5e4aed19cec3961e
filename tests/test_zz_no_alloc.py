"""The allocation-free backward entry point (m2rnn_backward_noalloc).

It serves callers that cannot call cudaMalloc (code inside a runtime that owns
all device memory, or paths where an allocation is not allowed): its scratch
lives in an array built into the library.  This file is collected last so that
a run stopping at the first failure has already run every other test.  It
passes alone in a fresh process and after the other tests (the first call on a
device sets up the array's address; later calls reuse it).
"""
import numpy as np
import pytest

from matrix_state_non_gb300.inputs import make_inputs
from oracle import backward as oracle_backward
from parity_util import GRAD_NAMES, TOL_BF16_REL, oracle_args, rel_fro

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "f", "W", "w_r")


def _case(B, N, T, K, C, seed):
    """Inputs, the forward's checkpoints, the workspace entry point's gradients
    and the oracle's, for one problem."""
    import torch

    from matrix_state_non_gb300 import binding
    inp = make_inputs(B, N, T, K, 64, "bf16", seed=seed, with_dy=True)
    d = binding.to_device(inp)
    dH = np.random.default_rng(seed + 100).standard_normal((B, N, K, 64)).astype(np.float32)
    dHd = torch.from_numpy(dH).cuda()
    fwd = binding.forward(*(d[n] for n in NAMES), ckpt_every=C)
    ws = binding.backward(*(d[n] for n in NAMES), d["dy"], dH_T=dHd, ckpt=fwd["ckpt"], ckpt_every=C)
    torch.cuda.synchronize()
    ws = {name: ws[name].cpu().numpy() for name in GRAD_NAMES}
    ref = oracle_backward(*oracle_args(inp), inp.exact["dy"], dH_T=dH)
    ora = {name: ref[name] for name in GRAD_NAMES}
    return dict(B=B, N=N, T=T, K=K, C=C, d=d, dH=dHd, ckpt=fwd["ckpt"], ws=ws, oracle=ora)


def _call(c, sync):
    import torch

    from matrix_state_non_gb300 import binding
    out = {name: torch.full(c["ws"][name].shape, float("nan"), device="cuda") for name in GRAD_NAMES}
    stream = torch.cuda.current_stream().cuda_stream
    st = binding.m2rnn_backward_noalloc(
        *(c["d"][n].data_ptr() for n in NAMES), c["d"]["dy"].data_ptr(), c["dH"].data_ptr(),
        c["ckpt"].data_ptr(), c["C"], *(out[name].data_ptr() for name in GRAD_NAMES),
        c["B"], c["T"], c["N"], c["K"], 64, binding.M2RNN_BF16, sync, stream)
    if st == binding.M2RNN_OK and not sync:
        st, detail = binding.m2rnn_backward_noalloc_status(stream)
        assert st == binding.M2RNN_OK, (binding.status_string(st), detail)
    assert st == binding.M2RNN_OK, binding.status_string(st)
    return {name: out[name].cpu().numpy() for name in GRAD_NAMES}


def _check(got, c, label):
    for name in GRAD_NAMES:
        assert np.all(np.isfinite(got[name])), (label, name)
        assert rel_fro(got[name], c["ws"][name]) <= TOL_BF16_REL, (label, name, "vs workspace path")
        assert rel_fro(got[name], c["oracle"][name]) <= TOL_BF16_REL, (label, name, "vs oracle")


def test_backward_noalloc_matches_workspace_entry_point_and_oracle():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    # A larger problem first, then a smaller one with other inputs (so scratch
    # left by the first call that the second wrongly read would show up), then
    # the first again: three calls in a row share the built-in scratch.
    big = _case(2, 2, 200, 64, 16, seed=31)
    small = _case(1, 3, 77, 32, 12, seed=47)
    _check(_call(big, sync=1), big, "first call")
    _check(_call(small, sync=0), small, "smaller problem, status read afterwards")
    _check(_call(big, sync=1), big, "first problem again")


def test_backward_noalloc_rejects_oversized_problem():
    from matrix_state_non_gb300 import binding
    # 1024 chains of 128 rows need 128 MiB of dW partials, more than the built-in scratch.
    st = binding.m2rnn_backward_noalloc(*([16] * 9), 16, *([16] * 6), 16, 1024, 64, 128, 64,
                                        binding.M2RNN_BF16, 0, None)
    assert st == binding.M2RNN_ERR_WORKSPACE
