"""Failure detection on the GPU without a GPU fault: a test hook withholds one
input tile, the consumers' bounded waits expire (about 2 s), the kernel
records a timeout in the workspace status block and returns, and the context
stays usable for the next call."""
import numpy as np
import pytest

from matrix_state_non_gb300.inputs import make_inputs
from oracle import forward as oracle_forward
from parity_util import TOL_BF16_REL, check_forward, gpu_forward, oracle_args, rel_fro

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "f", "W", "w_r")


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    from matrix_state_non_gb300 import binding
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    # K = 16 rows: one CTA per chain, no cluster peer left waiting.  The hook
    # lives in the warp-MMA forward (its waits use the same bounded helper as
    # every other kernel's).
    inp = make_inputs(1, 1, 200, 16, 64, "bf16", seed=3)
    d = binding.to_device(inp)
    with binding.kernel_family("mma"), binding.stall_tile_hook(1):
        out = binding.forward(*(d[n] for n in NAMES))
        st, detail = binding.sync_status(out["workspace"])
    assert st == binding.M2RNN_ERR_TIMEOUT, binding.status_string(st)
    # The consumers (input tile), the producer (free stage) and the reducer
    # (readout tile) all wait on the withheld tile; whichever gives up first
    # is recorded: any forward-kernel wait site (codes 1xx).
    assert detail // 100 == 1, detail
    got = gpu_forward(inp)  # the same context keeps working
    y_ref, H_ref = oracle_forward(*oracle_args(inp))
    check_forward(got, y_ref, H_ref, "bf16")


@pytest.mark.parametrize("V", [64, 16])
def test_query_outside_fp16_range_is_reported(V):
    """The warp-MMA forwards with readout warps (V = 64, and V = 16 with
    K <= 64) read out y with q re-encoded as fp16; a q entry of magnitude
    65536 or more is reported through the status block (location 302), and
    the next call on the same context is clean."""
    import torch
    from matrix_state_non_gb300 import binding
    from matrix_state_non_gb300.inputs import f32_to_bf16_bits
    inp = make_inputs(1, 2, 40, 64, V, "bf16", seed=13)
    inp.store["q"] = inp.store["q"].copy()
    inp.store["q"][0, 33, 1, 7] = f32_to_bf16_bits(np.array([-70000.0], dtype=np.float32))[0]
    d = binding.to_device(inp)
    out = binding.forward(*(d[n] for n in NAMES))
    st, detail = binding.sync_status(out["workspace"])
    assert st == binding.M2RNN_ERR_DEVICE and detail == 302, (binding.status_string(st), detail)
    # 65280, the largest bf16 magnitude below the limit, is accepted: no
    # error, finite y, and y within the relative tolerance (its absolute
    # error scales with that q, so only the relative bar applies).
    edge = make_inputs(1, 2, 40, 64, V, "bf16", seed=14)
    edge.store["q"] = edge.store["q"].copy()
    edge.store["q"][0, 5, 0, 3] = f32_to_bf16_bits(np.array([65280.0], dtype=np.float32))[0]
    edge.exact["q"] = edge.exact["q"].copy()
    edge.exact["q"][0, 5, 0, 3] = 65280.0
    d = binding.to_device(edge)
    out = binding.forward(*(d[n] for n in NAMES))
    st, detail = binding.sync_status(out["workspace"])
    assert st == binding.M2RNN_OK, (binding.status_string(st), detail)
    y = out["y"].cpu().numpy()
    assert np.isfinite(y).all()
    y_ref, _ = oracle_forward(*oracle_args(edge))
    assert rel_fro(y, y_ref) <= TOL_BF16_REL, rel_fro(y, y_ref)
    torch.cuda.synchronize()


@pytest.mark.parametrize("K,V", [(64, 64), (64, 16), (128, 128)])
def test_weight_outside_fp16_range_is_reported(K, V):
    """The tensor-core kernels take W re-encoded as fp16; an entry of W that
    fp16 cannot hold (|W| >= 65520) is reported through the status block
    (M2RNN_ERR_DEVICE at the input-check site), not silently turned into
    infinities.  The run itself completes; the next call is clean."""
    import torch
    from matrix_state_non_gb300 import binding
    from matrix_state_non_gb300.inputs import f32_to_bf16_bits
    inp = make_inputs(1, 2, 40, K, V, "bf16", seed=11)
    inp.store["W"] = inp.store["W"].copy()
    inp.store["W"][1, 3, 5] = f32_to_bf16_bits(np.array([70000.0], dtype=np.float32))[0]
    d = binding.to_device(inp)
    out = binding.forward(*(d[n] for n in NAMES))
    st, detail = binding.sync_status(out["workspace"])
    assert st == binding.M2RNN_ERR_DEVICE and detail == 301, (binding.status_string(st), detail)
    # A W inside the range on the same context: no error, and the oracle agrees.
    good = make_inputs(1, 2, 40, K, V, "bf16", seed=12)
    got = gpu_forward(good)
    y_ref, H_ref = oracle_forward(*oracle_args(good))
    check_forward(got, y_ref, H_ref, "bf16", label=("after range error", K, V))
    torch.cuda.synchronize()
