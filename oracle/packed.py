"""Adapters from the library's packed tensors to the oracle's plain arrays.

TEST INFRASTRUCTURE, like the rest of this package. Converts torch tensors to exact
float64 numpy arrays and turns the packed expert weights (W13 [E, R, d] with gate
rows then up rows, W2 [E, d, F]) into the math-layout matrices the oracle's expert
functions take: W_gate = W13[e, :F].T, W_up = W13[e, F:].T, W_down = W2[e].T. No
arithmetic of the layer lives here.
"""
from __future__ import annotations

import numpy as np

from oracle import moe_oracle as orc


def f64(t):
    """Exact float64 numpy copy of a tensor or array (None stays None)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def expert_fn(kind: str, W13, W2, F: int, faithful: bool = False, cache=None, fp8_up: bool = False,
              fp8_h: bool = False):
    """Expert_e(X) for the oracle, reading expert e's packed weights on demand.

    ``cache`` (a dict) keeps each expert's float64 weights after first use. With
    ``fp8_up`` the up-projection weights are the oracle's row-wise e4m3 quantization of
    W13[e] (one scale per output channel), as the FP8 expert GEMM uses them. With
    ``fp8_h`` the hidden activation goes through ``fp8_hidden`` and W2[e] is quantized
    per output channel (per row of W2[e] [d, F]): the FP8 down projection.
    """
    if kind == "identity":
        return lambda e, X: X

    def weights(e):
        if cache is not None and e in cache:
            return cache[e]
        w13, w2 = f64(W13[e]), f64(W2[e])
        if fp8_up:
            w13 = orc.quantize_fp8_rows(w13)["deq"]
        if fp8_h:
            w2 = orc.quantize_fp8_rows(w2)["deq"]
        w = (w13, w2)
        if cache is not None:
            cache[e] = w
        return w

    hidden = orc.fp8_hidden if fp8_h else None
    if kind == "relu":
        def fn(e, X):
            w13, w2 = weights(e)
            return orc.expert_relu(X, w13.T, w2.T, hidden=hidden)
    elif kind == "swiglu":
        def fn(e, X):
            w13, w2 = weights(e)
            return orc.expert_swiglu(X, w13[:F].T, w13[F:].T, w2.T, faithful=faithful, hidden=hidden)
    else:
        raise ValueError(kind)
    return fn


def run_oracle(w, inp: dict, capacity="auto", faithful: bool = False, cache=None) -> dict:
    """Oracle forward of workload ``w`` (sizes, expert kind, capacity) on tensors ``inp``."""
    if capacity == "auto":
        capacity = orc.expert_capacity(w.T, w.k, w.E, w.capacity_factor, w.min_capacity)
    fn = expert_fn(w.expert, inp.get("W13"), inp.get("W2"), w.F, faithful=faithful, cache=cache,
                   fp8_up=getattr(w, "dispatch_dtype", "act") == "fp8_gemm",
                   fp8_h=getattr(w, "precision", "") == "fp8_h")
    return orc.moe_forward(f64(inp["x"]), f64(inp["Wg"]), w.k, fn, capacity=capacity,
                           bias=f64(inp.get("bias")), D=w.D, n_shared=getattr(w, "n_shared", 0),
                           drop_policy=getattr(w, "drop_policy", "token"), layout=getattr(w, "layout", "packed"),
                           n_groups=getattr(w, "n_groups", 0), topk_groups=getattr(w, "topk_groups", 0),
                           dispatch_dtype=getattr(w, "dispatch_dtype", "act"))
