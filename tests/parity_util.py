"""Helpers shared by the GPU parity tests: run the library on seeded inputs and
compare with the float64 oracle at the stated tolerances."""
import numpy as np

# bf16-operand / fp32-state runs: max-abs <= 3e-2 on y, relative Frobenius
# <= 1e-2 on y, the final state and every gradient.  All-fp32 runs: 1e-4.
TOL_BF16_MAXABS_Y = 3e-2
TOL_BF16_REL = 1e-2
TOL_F32 = 1e-4

IN_NAMES = ("q", "k", "v", "f", "W", "w_r")
GRAD_NAMES = ("dq", "dk", "dv", "df", "dW", "dw_r")


def rel_fro(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return num
    return num / den


def max_abs(x, ref):
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64)))) if np.size(ref) else 0.0


def _cuda_f32(x):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def gpu_forward(inp, ckpt_every=0, H_0=None):
    import torch
    from matrix_state_non_gb300 import binding
    d = binding.to_device(inp)
    out = binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=ckpt_every, H_0=_cuda_f32(H_0))
    st, detail = binding.sync_status(out["workspace"])
    assert st == binding.M2RNN_OK, (binding.status_string(st), detail)
    torch.cuda.synchronize()
    res = {"y": out["y"].cpu().numpy(), "H_T": out["H_T"].cpu().numpy()}
    if "ckpt" in out:
        res["ckpt"] = out["ckpt"].cpu().numpy()
    return res


def gpu_backward(inp, dH_T=None, ckpt_every=16, use_fwd_ckpt=False, H_0=None, want_dH0=False,
                 state_grad_clip=0.0, stash=False):
    """stash: the forward also leaves its Z stash, which the backward reads
    (implies the forward's checkpoints)."""
    import torch
    from matrix_state_non_gb300 import binding
    d = binding.to_device(inp)
    h0 = _cuda_f32(H_0)
    ckpt = z = None
    if use_fwd_ckpt or stash:
        fo = binding.forward(*(d[n] for n in IN_NAMES), ckpt_every=ckpt_every, H_0=h0, stash=stash)
        ckpt, z = fo["ckpt"], fo.get("z_stash")
    out = binding.backward(*(d[n] for n in IN_NAMES), d["dy"], dH_T=_cuda_f32(dH_T), H_0=h0,
                           want_dH0=want_dH0, ckpt=ckpt, ckpt_every=ckpt_every,
                           state_grad_clip=state_grad_clip, z_stash=z)
    st, detail = binding.sync_status(out["workspace"])
    assert st == binding.M2RNN_OK, (binding.status_string(st), detail)
    torch.cuda.synchronize()
    names = GRAD_NAMES + (("dH_0",) if want_dH0 else ())
    return {k: out[k].cpu().numpy() for k in names}


def oracle_args(inp, sl_b=slice(None), sl_n=slice(None)):
    e = inp.exact
    return [e["q"][sl_b, :, sl_n], e["k"][sl_b, :, sl_n], e["v"][sl_b, :, sl_n],
            e["f"][sl_b, :, sl_n], e["W"][sl_n], e["w_r"][sl_n]]


def check_forward(got, y_ref, H_ref, dtype, label=""):
    if dtype == "f32":
        assert max_abs(got["y"], y_ref) <= TOL_F32, (label, max_abs(got["y"], y_ref))
        assert rel_fro(got["y"], y_ref) <= TOL_F32, (label, rel_fro(got["y"], y_ref))
        assert max_abs(got["H_T"], H_ref) <= TOL_F32, (label, max_abs(got["H_T"], H_ref))
        assert rel_fro(got["H_T"], H_ref) <= TOL_F32, (label, rel_fro(got["H_T"], H_ref))
    else:
        assert max_abs(got["y"], y_ref) <= TOL_BF16_MAXABS_Y, (label, max_abs(got["y"], y_ref))
        assert rel_fro(got["y"], y_ref) <= TOL_BF16_REL, (label, rel_fro(got["y"], y_ref))
        assert rel_fro(got["H_T"], H_ref) <= TOL_BF16_REL, (label, rel_fro(got["H_T"], H_ref))


def check_grads(got, ref, dtype, label=""):
    tol = TOL_F32 if dtype == "f32" else TOL_BF16_REL
    for name in GRAD_NAMES + (("dH_0",) if "dH_0" in got else ()):
        r = rel_fro(got[name], ref[name])
        assert r <= tol, (label, name, r)
