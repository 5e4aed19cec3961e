"""C-ABI boundary checks that need no GPU: the library loads, exports every
function include/m2rnn.h declares, and rejects bad arguments before touching
the device (so these calls are safe on a host without a GPU)."""
import os
import re

import pytest

from matrix_state_non_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return binding.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "m2rnn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(m2rnn_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "m2rnn_forward" in names and "m2rnn_backward" in names
    for name in names:
        assert hasattr(lib, name), name


def test_host_helpers(lib):
    assert binding.m2rnn_version() >= 10000
    assert binding.status_string(binding.M2RNN_ERR_WORKSPACE) == "workspace missing or too small"
    assert binding.status_string(12345) == "unknown status"
    assert binding.m2rnn_checkpoint_count(4096, 32) == 127
    assert binding.m2rnn_checkpoint_count(64, 64) == 0
    assert binding.m2rnn_checkpoint_count(0, 4) == -1
    # forward families: tcgen05 for V=64 and V=128 bf16, warp MMA for V=16 bf16, fp32 CUDA cores otherwise
    assert binding.m2rnn_path(64, 64, binding.M2RNN_BF16) == 2   # V = 64 forward: the warp-MMA scan
    assert binding.m2rnn_path(128, 128, binding.M2RNN_BF16) == 1
    assert binding.m2rnn_path(64, 16, binding.M2RNN_BF16) == 2
    assert binding.m2rnn_path(16, 16, binding.M2RNN_F32) == 0
    assert binding.m2rnn_path(200, 64, binding.M2RNN_BF16) == binding.M2RNN_ERR_UNSUPPORTED
    assert binding.m2rnn_path(64, 64, 7) == binding.M2RNN_ERR_INVALID_ARG


def test_workspace_sizes(lib):
    assert binding.m2rnn_forward_workspace_size(2, 16384, 16, 64, 64, binding.M2RNN_BF16) == 256
    assert binding.m2rnn_forward_workspace_size(0, 16, 1, 64, 64, binding.M2RNN_BF16) == 0
    with_ck = binding.m2rnn_backward_workspace_size(4, 4096, 8, 64, 64, binding.M2RNN_BF16, 32, 1)
    without = binding.m2rnn_backward_workspace_size(4, 4096, 8, 64, 64, binding.M2RNN_BF16, 32, 0)
    assert without - with_ck >= 4 * 8 * 127 * 64 * 64 * 4  # the recomputed checkpoints
    assert binding.m2rnn_backward_workspace_size(4, 4096, 8, 64, 64, binding.M2RNN_BF16, 0, 1) == 0
    assert binding.m2rnn_backward_workspace_size(4, 4096, 8, 64, 64, binding.M2RNN_BF16, 5000, 1) == 0


P = 1 << 20  # a 16-byte-aligned fake address: never dereferenced by these calls


def fwd(**kw):
    a = dict(q=P, k=P, v=P, f=P, W=P, w_r=P, y=P, H_T=None, ckpt=None, C=0, B=1, T=8, N=1, K=64, V=64,
             dt=binding.M2RNN_BF16, ws=P, wsb=256, stream=None)
    a.update(kw)
    return binding.m2rnn_forward(a["q"], a["k"], a["v"], a["f"], a["W"], a["w_r"], a["y"], a["H_T"],
                                 a["ckpt"], a["C"], a["B"], a["T"], a["N"], a["K"], a["V"], a["dt"],
                                 a["ws"], a["wsb"], a["stream"])


def test_forward_rejects_bad_arguments_without_a_device(lib):
    assert fwd(q=None) == binding.M2RNN_ERR_INVALID_ARG
    assert fwd(y=None) == binding.M2RNN_ERR_INVALID_ARG
    assert fwd(k=P + 8) == binding.M2RNN_ERR_INVALID_ARG          # misaligned
    assert fwd(H_T=P + 4) == binding.M2RNN_ERR_INVALID_ARG
    assert fwd(B=0) == binding.M2RNN_ERR_INVALID_ARG
    assert fwd(T=-3) == binding.M2RNN_ERR_INVALID_ARG
    assert fwd(K=129) == binding.M2RNN_ERR_UNSUPPORTED
    assert fwd(V=256) == binding.M2RNN_ERR_UNSUPPORTED
    assert fwd(dt=9) == binding.M2RNN_ERR_INVALID_ARG
    assert fwd(ckpt=P, C=0) == binding.M2RNN_ERR_INVALID_ARG
    assert fwd(ws=None) == binding.M2RNN_ERR_WORKSPACE
    assert fwd(wsb=128) == binding.M2RNN_ERR_WORKSPACE


def bwd(**kw):
    a = dict(dH=None, ckpt=None, C=32, dq=P, B=1, T=8, N=1, K=64, V=64, dt=binding.M2RNN_BF16, ws=P,
             wsb=1 << 30)
    a.update(kw)
    return binding.m2rnn_backward(P, P, P, P, P, P, P, a["dH"], a["ckpt"], a["C"], a["dq"], P, P, P, P, P,
                                  a["B"], a["T"], a["N"], a["K"], a["V"], a["dt"], a["ws"], a["wsb"], None)


def test_backward_rejects_bad_arguments_without_a_device(lib):
    assert bwd(dq=None) == binding.M2RNN_ERR_INVALID_ARG
    assert bwd(dH=P + 2) == binding.M2RNN_ERR_INVALID_ARG
    assert bwd(C=0) == binding.M2RNN_ERR_INVALID_ARG
    assert bwd(C=4097) == binding.M2RNN_ERR_INVALID_ARG
    assert bwd(K=0) == binding.M2RNN_ERR_INVALID_ARG
    assert bwd(wsb=16) == binding.M2RNN_ERR_WORKSPACE
    assert bwd(ws=None) == binding.M2RNN_ERR_WORKSPACE


def test_state_entry_points_reject_bad_arguments_without_a_device(lib):
    # Misaligned initial state / state gradient, and a decode step without a state.
    st = binding.m2rnn_forward_state(P, P, P, P, P, P, P + 4, P, None, None, 0, None, 1, 8, 1, 1, 64, 64,
                                     binding.M2RNN_BF16, P, 1 << 20, None)
    assert st == binding.M2RNN_ERR_INVALID_ARG
    st = binding.m2rnn_forward_state(P, P, P, P, P, P, None, P, None, None, 0, None, 1, 8, 4, 2, 64, 64,
                                     binding.M2RNN_BF16, P, 1 << 20, None)
    assert st == binding.M2RNN_ERR_INVALID_ARG   # q/k heads must be 1 or N
    assert binding.m2rnn_backward_state_workspace_size(1, 8, 4, 3, 64, 64, binding.M2RNN_BF16, 14, 1) == 0
    shared = binding.m2rnn_backward_state_workspace_size(2, 8, 4, 1, 64, 64, binding.M2RNN_BF16, 14, 1)
    per_head = binding.m2rnn_backward_state_workspace_size(2, 8, 4, 4, 64, 64, binding.M2RNN_BF16, 14, 1)
    assert shared >= per_head + 2 * 4 * 2 * 8 * 4 * 64   # room for the per-head dq, dk
    common = dict(B=1, T=8, N=1, QK=1, K=64, V=64)
    st = binding.m2rnn_backward_state(P, P, P, P, P, P, None, P, None, None, 14, None, P, P, P, P, P, P,
                                      P + 8, 0.0, *common.values(), binding.M2RNN_BF16, P, 1 << 30, None)
    assert st == binding.M2RNN_ERR_INVALID_ARG
    for bad_clip in (-1.0, float("nan")):
        st = binding.m2rnn_backward_state(P, P, P, P, P, P, None, P, None, None, 14, None, P, P, P, P, P, P,
                                          None, bad_clip, *common.values(), binding.M2RNN_BF16, P,
                                          1 << 30, None)
        assert st == binding.M2RNN_ERR_INVALID_ARG
    st = binding.m2rnn_decode_step(None, P, P, P, P, P, P, P, 1, 1, 1, 64, 64, binding.M2RNN_BF16, P,
                                   1 << 20, None)
    assert st == binding.M2RNN_ERR_INVALID_ARG
    st = binding.m2rnn_decode_step(P, P, P, P, P, P, P, P, 1, 1, 1, 64, 200, binding.M2RNN_BF16, P,
                                   1 << 20, None)
    assert st == binding.M2RNN_ERR_UNSUPPORTED   # V above the supported 128


def test_gate_and_output_norm_entry_points_reject_bad_arguments_without_a_device(lib):
    bf = binding.M2RNN_BF16

    def fg(a=P, alpha=P, beta=P, N=2):
        return binding.m2rnn_forward_gated(P, P, P, a, alpha, beta, P, P, None, P, None, None, 0, None, 1, 8, N, N,
                                           64, 64, bf, P, 1 << 20, None)
    assert fg(a=None) == binding.M2RNN_ERR_INVALID_ARG
    assert fg(alpha=None) == binding.M2RNN_ERR_INVALID_ARG
    assert fg(beta=P + 4) == binding.M2RNN_ERR_INVALID_ARG

    def bg(dalpha=P, dbeta=P, a=P):
        return binding.m2rnn_backward_gated(P, P, P, a, P, P, P, P, None, P, None, None, 14, None, P, P, P, P, dalpha,
                                            dbeta, P, P, None, 0.0, 1, 8, 2, 2, 64, 64, bf, P, 1 << 30, None)
    assert bg(dalpha=None) == binding.M2RNN_ERR_INVALID_ARG
    assert bg(dbeta=P + 8) == binding.M2RNN_ERR_INVALID_ARG
    assert bg(a=None) == binding.M2RNN_ERR_INVALID_ARG

    assert binding.m2rnn_output_norm_backward_workspace_size(4, 4096, 8, 64) > 0
    assert binding.m2rnn_output_norm_backward_workspace_size(1, 8, 129, 128) == 0   # N V above 16384
    assert binding.m2rnn_output_norm_backward_workspace_size(0, 8, 8, 64) == 0
    assert binding.m2rnn_output_norm(P, P, P, -1.0, P, None, 1, 8, 8, 64, bf, None) == \
        binding.M2RNN_ERR_INVALID_ARG
    assert binding.m2rnn_output_norm(P, P, P, float("nan"), P, None, 1, 8, 8, 64, bf, None) == \
        binding.M2RNN_ERR_INVALID_ARG
    assert binding.m2rnn_output_norm(P, P + 2, P, 1e-6, P, None, 1, 8, 8, 64, bf, None) == \
        binding.M2RNN_ERR_INVALID_ARG
    assert binding.m2rnn_output_norm(P, P, P, 1e-6, P, None, 1, 8, 129, 128, bf, None) == \
        binding.M2RNN_ERR_UNSUPPORTED
    assert binding.m2rnn_output_norm_backward(P, P, P, P, 1e-6, P, P, P, 1, 8, 8, 64, bf, P, 16, None) == \
        binding.M2RNN_ERR_WORKSPACE
    assert binding.m2rnn_output_norm_backward(P, P, P, None, 1e-6, P, P, P, 1, 8, 8, 64, bf, P, 1 << 30,
                                              None) == binding.M2RNN_ERR_INVALID_ARG


def test_z_stash_rules_without_a_device(lib):
    bf = binding.M2RNN_BF16
    assert binding.m2rnn_z_stash_size(4, 4096, 8, 64, 64, bf) == 4 * 4096 * 8 * 64 * 64 * 2
    assert binding.m2rnn_z_stash_size(1, 8, 1, 128, 128, bf) == 0            # V = 128: no stash
    assert binding.m2rnn_z_stash_size(1, 8, 1, 64, 64, binding.M2RNN_F32) == 0
    assert binding.m2rnn_z_stash_size(1, 8, 1, 40, 64, bf) == 0              # K not a multiple of 16

    assert binding.m2rnn_z_stash_size(2, 8, 4, 64, 16, bf) == 2 * 8 * 4 * 64 * 16 * 2   # V = 16 too

    def fs(V=64, z=P, K=64):
        return binding.m2rnn_forward_state(P, P, P, P, P, P, None, P, None, None, 0, z, 1, 8, 1, 1, K, V, bf, P,
                                           1 << 20, None)
    assert fs(V=128) == binding.M2RNN_ERR_UNSUPPORTED
    assert fs(K=40, V=16) == binding.M2RNN_ERR_UNSUPPORTED   # K not a multiple of 16
    assert fs(V=32) == binding.M2RNN_ERR_UNSUPPORTED
    assert fs(z=P + 8) == binding.M2RNN_ERR_INVALID_ARG

    def bs(T=64, ckpt=None, C=14, z=P):
        return binding.m2rnn_backward_state(P, P, P, P, P, P, None, P, None, ckpt, C, z, P, P, P, P, P, P, None,
                                            0.0, 1, T, 1, 1, 64, 64, bf, P, 1 << 30, None)
    assert bs() == binding.M2RNN_ERR_INVALID_ARG          # T > ckpt_every needs the forward's checkpoints
    assert bs(C=21, ckpt=P) == binding.M2RNN_ERR_UNSUPPORTED   # longer than the backward's chunk cache
    assert bs(z=P + 4, ckpt=P) == binding.M2RNN_ERR_INVALID_ARG

    def bs16(K=64, C=14):
        return binding.m2rnn_backward_state(P, P, P, P, P, P, None, P, None, P, C, P, P, P, P, P, P, P, None,
                                            0.0, 1, 64, 1, 1, K, 16, bf, P, 1 << 30, None)
    assert bs16(K=128, C=17) == binding.M2RNN_ERR_UNSUPPORTED   # over the V = 16 chunk limit for K > 64
    assert bs16(K=64, C=33) == binding.M2RNN_ERR_UNSUPPORTED


def test_noalloc_backward_rejects_unsupported_shapes_without_a_device(lib):
    def call(**kw):
        a = dict(C=16, B=1, T=64, N=1, K=64, V=64, dt=binding.M2RNN_BF16, ckpt=P)
        a.update(kw)
        return binding.m2rnn_backward_noalloc(P, P, P, P, P, P, P, None, a["ckpt"], a["C"], P, P, P, P, P, P,
                                              a["B"], a["T"], a["N"], a["K"], a["V"], a["dt"], 0, None)
    assert call(V=128) == binding.M2RNN_ERR_UNSUPPORTED
    assert call(dt=binding.M2RNN_F32) == binding.M2RNN_ERR_UNSUPPORTED
    assert call(C=21) == binding.M2RNN_ERR_UNSUPPORTED            # longer than the TMEM chunk cache
    assert call(ckpt=None) == binding.M2RNN_ERR_INVALID_ARG      # T > C needs the forward's checkpoints
    assert call(B=4096, N=1024) == binding.M2RNN_ERR_WORKSPACE   # exceeds the built-in scratch


def test_kernel_family_option(lib):
    with binding.kernel_family("tcgen05"):
        assert binding.m2rnn_path(64, 64, binding.M2RNN_BF16) == 1
    with binding.kernel_family("simt"):
        assert binding.m2rnn_path(64, 64, binding.M2RNN_BF16) == 0
    with binding.kernel_family("mma"):
        assert binding.m2rnn_path(64, 64, binding.M2RNN_BF16) == 2
        assert binding.m2rnn_path(128, 128, binding.M2RNN_BF16) == 1  # no warp-MMA kernel for V=128
    assert binding.m2rnn_path(64, 64, binding.M2RNN_BF16) == 2      # the automatic choice is back
    st, _ = binding.m2rnn_set_option(binding.M2RNN_OPT_KERNEL_FAMILY, 3)
    assert st == binding.M2RNN_ERR_INVALID_ARG
    st, _ = binding.m2rnn_set_option(99, 0)
    assert st == binding.M2RNN_ERR_INVALID_ARG
    with binding.stall_tile_hook(4):
        st, prev = binding.m2rnn_set_option(binding.M2RNN_OPT_TEST_STALL_TILE, 4)
        assert st == binding.M2RNN_OK and prev == 4
    st, prev = binding.m2rnn_set_option(binding.M2RNN_OPT_TEST_STALL_TILE, -1)
    assert st == binding.M2RNN_OK and prev == -1


def test_options_start_from_the_environment(root_dir):
    """The switches take their first values from M2RNN_KERNEL and
    M2RNN_TEST_STALL_TILE, read once (checked in a fresh process)."""
    import subprocess
    import sys
    code = ("from matrix_state_non_gb300 import binding as b; "
            "print(b.m2rnn_path(64, 64, b.M2RNN_BF16), b.m2rnn_set_option(b.M2RNN_OPT_TEST_STALL_TILE, -1)[1])")
    env = dict(os.environ, M2RNN_KERNEL="simt", M2RNN_TEST_STALL_TILE="3")
    out = subprocess.run([sys.executable, "-c", code], cwd=root_dir, env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["0", "3"]


def test_fp16_operand_range_limits():
    """The range limits the kernels check for their fp16 operands (W: the
    location-301 check; q in the warp-MMA readouts: location 302, which
    compares the bf16 magnitude bits with 0x4780) are where fp16 stops
    holding the value: 0x4780 is bf16 65536, which fp16 rounds to infinity,
    while 65280, the bf16 value just below, is exact in fp16; for W (any
    real input) fp16 overflows from 65520 on."""
    import numpy as np
    bf16_bits_to_f32 = lambda b: np.array([b << 16], dtype=np.uint32).view(np.float32)[0]
    assert bf16_bits_to_f32(0x4780) == 65536.0
    assert bf16_bits_to_f32(0x477F) == 65280.0
    with np.errstate(over="ignore"):
        assert np.isinf(np.float16(np.float32(65536.0)))
        assert np.float16(np.float32(65280.0)) == 65280.0
        assert np.isinf(np.float16(np.float32(65520.0)))
        assert np.isfinite(np.float16(np.float32(65519.0)))
    # Every bf16 magnitude pattern below 0x4780 is finite in fp16, and none
    # at or above it (0x7F80 and up are infinities and NaNs).
    bits = np.arange(0x0000, 0x7F80, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    with np.errstate(over="ignore"):
        finite = np.isfinite(vals.astype(np.float16))
    assert finite[bits < 0x4780].all() and not finite[bits >= 0x4780].any()
