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
from parity_util import GRAD_NAMES, TOL_BF16_REL, rel_fro

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "f", "W", "w_r")


def test_backward_noalloc_matches_workspace_entry_point():
    import torch

    from matrix_state_non_gb300 import binding

    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    B, N, T, K, V, C = 2, 2, 200, 64, 64, 16
    inp = make_inputs(B, N, T, K, V, "bf16", seed=31, with_dy=True)
    d = binding.to_device(inp)
    dH = torch.from_numpy(np.random.default_rng(2).standard_normal((B, N, K, V)).astype(np.float32)).cuda()
    fwd = binding.forward(*(d[n] for n in NAMES), ckpt_every=C)
    ref = binding.backward(*(d[n] for n in NAMES), d["dy"], dH_T=dH, ckpt=fwd["ckpt"], ckpt_every=C)
    torch.cuda.synchronize()
    ref = {name: ref[name].cpu().numpy() for name in GRAD_NAMES}
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row share (and reuse) the built-in scratch
        out = {name: torch.full(ref[name].shape, float("nan"), device="cuda") for name in GRAD_NAMES}
        st = binding.m2rnn_backward_noalloc(
            *(d[n].data_ptr() for n in NAMES), d["dy"].data_ptr(), dH.data_ptr(),
            fwd["ckpt"].data_ptr(), C, *(out[name].data_ptr() for name in GRAD_NAMES),
            B, T, N, K, V, binding.M2RNN_BF16, 1, stream)
        assert st == binding.M2RNN_OK, (call, binding.status_string(st))
        for name in GRAD_NAMES:
            got = out[name].cpu().numpy()
            assert np.all(np.isfinite(got)), (call, name)
            assert rel_fro(got, ref[name]) <= TOL_BF16_REL, (call, name, rel_fro(got, ref[name]))


def test_backward_noalloc_rejects_oversized_problem():
    from matrix_state_non_gb300 import binding
    # 1024 chains of 128 rows need 128 MiB of dW partials, more than the built-in scratch.
    st = binding.m2rnn_backward_noalloc(*([16] * 9), 16, *([16] * 6), 16, 1024, 64, 128, 64,
                                        binding.M2RNN_BF16, 0, None)
    assert st == binding.M2RNN_ERR_WORKSPACE
