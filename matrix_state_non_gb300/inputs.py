"""Seeded synthetic inputs for the M2RNN scans.

This module is shared by the CUDA path's callers (tests, bench) and by the
float64 oracle's callers.  It draws random numbers and rounds them to the
storage dtype; it holds none of the recurrence's arithmetic.

Distributions follow the workload description of the M2RNN recurrence
(Eq. 10-12 of "M2RNN: Non-Linear RNNs with Matrix-Valued States for Scalable
Language Modeling"): q, k ~ N(0,1)/sqrt(K); v ~ N(0,1); f = sigmoid(N(2,1)) per
(b, t, head); W ~ N(0, 1/V) per head; w_r ~ N(0,1); upstream dy ~ N(0,1).

Generator: numpy PCG64 seeded with the integer seed; draws in the fixed order
q, k, v, f, W, w_r, dy, each as float64 of the full shape.  bf16 storage
rounds float64 -> float32 (round to nearest even) -> bf16 (round to nearest
even on the float32 bits).  Both sides consume exactly the rounded values.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# The named workloads: shapes, storage dtype, whether the backward runs, seed.
WORKLOADS = {
    "tiny_f32": dict(B=1, N=2, T=64, K=16, V=16, dtype="f32", backward=False, seed=0,
                     desc="tiny fp32 forward B=1 heads=2 T=64 K=16 V=16"),
    "fwd_bf16_k64": dict(B=4, N=8, T=2048, K=64, V=64, dtype="bf16", backward=False, seed=1,
                         desc="bf16 forward B=4 heads=8 T=2048 K=64 V=64"),
    "fwd_bf16_k128": dict(B=8, N=16, T=4096, K=128, V=128, dtype="bf16", backward=False, seed=2,
                          desc="bf16 wide-head forward B=8 heads=16 T=4096 K=128 V=128"),
    "fwd_bf16_16k": dict(B=2, N=16, T=16384, K=64, V=64, dtype="bf16", backward=False, seed=3,
                         desc="bf16 long-context forward B=2 heads=16 T=16384 K=64 V=64"),
    "fwdbwd_bf16_k64": dict(B=4, N=8, T=4096, K=64, V=64, dtype="bf16", backward=True, seed=4,
                            desc="bf16 forward+backward B=4 heads=8 T=4096 K=64 V=64"),
    # The wide-head shape trained: forward + backward at B=8 heads=16 K=V=128
    # (the forward-only wide-head workload's batch, a quarter of its length).
    "fwdbwd_bf16_k128": dict(B=8, N=16, T=1024, K=128, V=128, dtype="bf16", backward=True, seed=6,
                             desc="bf16 wide-head forward+backward B=8 heads=16 T=1024 K=128 V=128"),
    # Multi-value heads (the pages' K = 64, V = 16 per head, one q/k shared by
    # every head) at the forward+backward workload's batch and length.
    "mv_bf16_k64v16": dict(B=4, N=16, T=4096, K=64, V=16, dtype="bf16", backward=True, seed=5,
                           shared_qk=True,
                           desc="bf16 multi-value forward+backward B=4 heads=16 T=4096 K=64 V=16, shared q/k"),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even), returned as uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    # NaN is never produced by the distributions above; keep the rounding plain.
    bias = ((bits >> 16) & 1) + 0x7FFF
    out = ((bits + bias) >> 16) & 0xFFFF
    return out.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    u32 = (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16)
    return u32.view(np.float32).astype(np.float64)


def round_to_dtype(x64: np.ndarray, dtype: str):
    """Return (storage array, exact float64 value of the stored data)."""
    x32 = x64.astype(np.float32)
    if dtype == "f32":
        return x32, x32.astype(np.float64)
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x32)
        return bits, bf16_bits_to_f64(bits)
    raise ValueError(f"unknown dtype {dtype!r}")


@dataclasses.dataclass
class M2RNNInputs:
    """One batch of inputs in both forms.

    ``store[name]`` is the array handed to the library (float32, or uint16 bf16
    bit patterns); ``exact[name]`` is its exact float64 value, which is what the
    oracle consumes.  Layouts: q, k [B,T,N,K]; v [B,T,N,V]; f [B,T,N];
    W [N,V,V]; w_r [N,V]; dy [B,T,N,V] (float32 in both dtypes).
    """

    B: int
    N: int
    T: int
    K: int
    V: int
    dtype: str
    store: dict
    exact: dict


def make_inputs(B: int, N: int, T: int, K: int, V: int, dtype: str = "bf16",
                seed: int = 0, with_dy: bool = False,
                f_mode: Optional[str] = None) -> M2RNNInputs:
    """Draw one seeded batch of inputs with the workload distributions.

    ``f_mode`` overrides the gate for special-case tests: "ones" (f = 1),
    "zeros" (f = 0); None keeps sigmoid(N(2,1)).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    raw = {}
    raw["q"] = rng.standard_normal((B, T, N, K)) / np.sqrt(K)
    raw["k"] = rng.standard_normal((B, T, N, K)) / np.sqrt(K)
    raw["v"] = rng.standard_normal((B, T, N, V))
    g = rng.standard_normal((B, T, N)) + 2.0
    raw["f"] = 1.0 / (1.0 + np.exp(-g))
    raw["W"] = rng.standard_normal((N, V, V)) / np.sqrt(V)
    raw["w_r"] = rng.standard_normal((N, V))
    if with_dy:
        raw["dy"] = rng.standard_normal((B, T, N, V))
    if f_mode == "ones":
        raw["f"] = np.ones((B, T, N))
    elif f_mode == "zeros":
        raw["f"] = np.zeros((B, T, N))
    elif f_mode is not None:
        raise ValueError(f"unknown f_mode {f_mode!r}")
    store, exact = {}, {}
    for name in ("q", "k", "v", "f", "W", "w_r"):
        store[name], exact[name] = round_to_dtype(raw[name], dtype)
    if with_dy:
        store["dy"], exact["dy"] = round_to_dtype(raw["dy"], "f32")
    return M2RNNInputs(B, N, T, K, V, dtype, store, exact)


def make_workload(name: str, seed: Optional[int] = None) -> M2RNNInputs:
    """Inputs of one of the named workloads (seed defaults to the workload's own)."""
    w = WORKLOADS[name]
    inp = make_inputs(w["B"], w["N"], w["T"], w["K"], w["V"], w["dtype"],
                      seed=w["seed"] if seed is None else seed, with_dy=w["backward"])
    if w.get("shared_qk"):  # one q/k for every head: keep head 0 of the drawn q, k
        for name_ in ("q", "k"):
            inp.store[name_] = np.ascontiguousarray(inp.store[name_][:, :, :1])
            inp.exact[name_] = np.ascontiguousarray(inp.exact[name_][:, :, :1])
    return inp


def from_exact(exact: dict, dtype: str) -> M2RNNInputs:
    """Wrap hand-built float64 inputs (already representable in ``dtype``)."""
    q = exact["q"]
    B, T, N, K = q.shape
    V = exact["v"].shape[-1]
    store, ex = {}, {}
    for name, arr in exact.items():
        dt = "f32" if name in ("dy", "dH_T") else dtype
        s, e = round_to_dtype(np.asarray(arr, dtype=np.float64), dt)
        if not np.array_equal(e, np.asarray(arr, dtype=np.float64)):
            raise ValueError(f"{name} is not exactly representable in {dt}")
        store[name], ex[name] = s, e
    return M2RNNInputs(B, N, T, K, V, dtype, store, ex)


def make_gate_inputs(B: int, T: int, N: int, dtype: str = "bf16", seed: int = 0):
    """Forget-gate parameters: the pre-activation a [B,T,N] ~ N(0, 1) in the
    storage dtype, and per head alpha ~ U(0.5, 2), beta ~ N(-2, 0.5) in fp32
    (so that a + beta centres where the f distribution above centres).
    Returns (store, exact) dicts with keys a, alpha, beta."""
    rng = np.random.default_rng(seed)
    raw = {"a": rng.standard_normal((B, T, N)),
           "alpha": rng.uniform(0.5, 2.0, N),
           "beta": rng.standard_normal(N) * 0.5 - 2.0}
    store, exact = {}, {}
    store["a"], exact["a"] = round_to_dtype(raw["a"], dtype)
    for name in ("alpha", "beta"):
        store[name], exact[name] = round_to_dtype(raw[name], "f32")
    return store, exact


def make_norm_inputs(B: int, T: int, N: int, V: int, dtype: str = "bf16", seed: int = 0):
    """Output-path inputs: a readout y [B,T,N,V] ~ N(0, 1/4) (fp32), the output
    gate g [B,T,N,V] ~ N(0, 1) in the storage dtype, the per-channel weight
    w [N,V] ~ 1 + N(0, 1/100) and the upstream gradient dout ~ N(0, 1) (fp32).
    Returns (store, exact) dicts with keys y, g, w, dout."""
    rng = np.random.default_rng(seed)
    raw = {"y": rng.standard_normal((B, T, N, V)) * 0.5,
           "g": rng.standard_normal((B, T, N, V)),
           "w": 1.0 + rng.standard_normal((N, V)) * 0.1,
           "dout": rng.standard_normal((B, T, N, V))}
    store, exact = {}, {}
    for name in ("y", "w", "dout"):
        store[name], exact[name] = round_to_dtype(raw[name], "f32")
    store["g"], exact["g"] = round_to_dtype(raw["g"], dtype)
    return store, exact
