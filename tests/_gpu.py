"""GPU-side test glue: runs the library through its C ABI and compares with the oracle.

Tolerances (floating point):
  * layer output y and expert outputs: max |gpu - exact| <= tol * rms(exact) + half an
    ulp of the activation dtype at the exact value, tol = 2e-2 (bf16) or 1e-4 (fp32).
    The half-ulp term is the representation error of the output format itself: no
    result delivered in bf16 can be closer to the exact value than that, so the
    relative tolerance is read as bounding the arithmetic (fp32 accumulation, the
    bf16 rounding of h and of the expert outputs) on top of it.
  * gates: |gpu - exact| <= 2e-6 (fp32 logits carry ~1e-7 absolute error from a
    d-long dot product summed in 256-term pieces; exp and the division add a few
    ulp).
Integer and index outputs (top-k ids away from near ties, counts, offsets, the
permutation, drop lists, dispatched rows) are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as orc
from routing_dispatch_combine_moe_b300 import abi
from tests._harness import expert_fn, f64

TOL = {"bf16": 2e-2, "f32": 1e-4}
GATE_TOL = 2e-6


def half_ulp(v: np.ndarray, act: str) -> np.ndarray:
    """Half an ulp of the activation dtype at |v| (bf16: 8 significant bits, fp32: 24)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-38)))
    bits = 8 if act == "bf16" else 24
    return 2.0 ** (e - bits)


def rms(v) -> float:
    v = np.asarray(v, np.float64)
    return float(np.sqrt(np.mean(v * v))) if v.size else 0.0


def check_close(got, exact, act: str, what: str, tol: float | None = None) -> float:
    """Asserts the float tolerance; returns the raw max|err| / rms(exact)."""
    tol = TOL[act] if tol is None else tol
    got = f64(got)
    exact = np.asarray(exact, np.float64)
    assert got.shape == exact.shape, (what, got.shape, exact.shape)
    r = rms(exact)
    err = np.abs(got - exact)
    bound = tol * r + half_ulp(exact, act)
    bad = err > bound
    assert not np.isnan(got).any(), f"{what}: NaN in GPU output"
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} elements beyond {tol}*rms + half-ulp; worst at {i}: "
                             f"gpu={got[i]!r} exact={exact[i]!r} err={err[i]:.3e} bound={bound[i]:.3e} rms={r:.3e}")
    return float(err.max() / r) if r > 0 else 0.0


class StageBuffers:
    """Output buffers of the four stage entry points, filled with sentinels."""

    def __init__(self, w, cfg, device="cuda"):
        A = w.T * w.slots
        N = w.n_experts
        i32 = dict(dtype=torch.int32, device=device)
        self.cfg = cfg
        self.topk_idx = torch.full((w.T, w.slots), -7, **i32)
        self.topk_gate = torch.full((w.T, w.slots), float("nan"), dtype=torch.float32, device=device)
        self.counts_routed = torch.full((N,), -7, **i32)
        self.counts_kept = torch.full((N,), -7, **i32)
        self.offsets = torch.full((N + 1,), -7, **i32)
        self.rank_offsets = torch.full((w.D + 1,), -7, **i32)
        self.pos = torch.full((A,), -7, **i32)
        self.row_src = torch.full((A,), -7, **i32)
        self.drop_list = torch.full((A,), -7, **i32)
        self.n_dropped = torch.full((1,), -7, **i32)
        self.xperm = torch.full((A, w.d), float("nan"), dtype=w.torch_act, device=device)
        self.h = torch.full((A, max(abi.hidden_cols(cfg), 1)), float("nan"), dtype=w.torch_act, device=device)
        self.out = torch.full((A, w.d), float("nan"), dtype=abi.out_dtype(cfg), device=device)
        self.out_act = "f32" if abi.out_dtype(cfg) == torch.float32 else "bf16"
        self.y = torch.full((w.T, w.d), float("nan"), dtype=w.torch_act, device=device)
        nr = abi.moe_route_workspace_bytes(cfg)
        self.ws_route = torch.zeros(nr, dtype=torch.uint8, device=device) if nr else None
        self.ws_dispatch = torch.zeros(abi.moe_dispatch_workspace_bytes(cfg), dtype=torch.uint8, device=device)
        self.ws_ffn = torch.zeros(abi.moe_ffn_workspace_bytes(cfg), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def dmap(self):
        return abi.dispatch_map(self.counts_routed, self.counts_kept, self.offsets, self.rank_offsets, self.pos,
                                self.row_src, self.drop_list, self.n_dropped)

    def route(self, inp):
        abi.moe_route(self.cfg, inp["x"], inp["Wg"], inp.get("bias"), self.topk_idx, self.topk_gate, self.ws_route)

    def dispatch(self, inp, topk_idx=None):
        abi.moe_dispatch(self.cfg, inp["x"], self.topk_idx if topk_idx is None else topk_idx, self.dmap(),
                         self.xperm, self.ws_dispatch)

    def ffn(self, inp):
        abi.moe_expert_ffn(self.cfg, self.xperm, self.offsets, inp["W13"], inp["W2"], self.h, self.out, self.ws_ffn)

    def combine(self, out=None):
        abi.moe_combine(self.cfg, self.out if out is None else out, self.topk_gate, self.pos, self.y, self.status)

    def dispatch_status(self) -> int:
        return abi.moe_read_status(self.ws_dispatch.data_ptr())

    def ffn_status(self) -> int:
        return abi.moe_read_status(self.ws_ffn.data_ptr())


def cpu(t):
    return t.detach().cpu()


def check_route(w, inp, bufs, H=None) -> dict:
    """Top-k ids exact away from near ties; gates within GATE_TOL. Returns stats."""
    if H is None:
        H = orc.router_logits(f64(inp["x"]), f64(inp["Wg"]), f64(inp.get("bias")))
    idx_o = orc.keep_topk(H, w.k)
    G_o = orc.kept_softmax(H, idx_o)
    set_tie, order_tie = orc.near_tie_flags(H, w.k)
    tie = set_tie | order_tie
    idx_all = cpu(bufs.topk_idx).numpy()
    G_all = cpu(bufs.topk_gate).numpy().astype(np.float64)
    S = getattr(w, "n_shared", 0)
    if S:  # shared slots follow the routed ones: experts E.., gate 1
        assert np.all(idx_all[:, w.k:] == w.E + np.arange(S)) and np.all(G_all[:, w.k:] == 1.0)
    idx_g, G_g = idx_all[:, :w.k], G_all[:, :w.k]
    mismatch = (idx_g != idx_o).any(axis=1)
    assert not (mismatch & ~tie).any(), \
        f"top-k differs on {int((mismatch & ~tie).sum())} tokens without a near tie, e.g. {np.nonzero(mismatch & ~tie)[0][:5]}"
    ok = ~mismatch
    gerr = np.abs(G_g[ok] - G_o[ok]).max() if ok.any() else 0.0
    assert gerr <= GATE_TOL, f"gate error {gerr:.3e} > {GATE_TOL}"
    assert np.all((idx_g >= 0) & (idx_g < w.E))
    return dict(near_ties=int(tie.sum()), flipped=int(mismatch.sum()), gate_err=float(gerr), H=H, idx=idx_o, G=G_o)


def check_dispatch(w, inp, bufs, capacity) -> dict:
    """Stage check on the GPU's own top-k: every routing-map array bit-exact, rows copied exactly."""
    idx_g = cpu(bufs.topk_idx).numpy().astype(np.int64)
    d = orc.dispatch(idx_g, w.n_experts, capacity, w.D, capped_experts=w.E)
    np.testing.assert_array_equal(cpu(bufs.counts_routed).numpy(), d["counts_routed"])
    np.testing.assert_array_equal(cpu(bufs.counts_kept).numpy(), d["counts_kept"])
    np.testing.assert_array_equal(cpu(bufs.offsets).numpy(), d["offsets"])
    np.testing.assert_array_equal(cpu(bufs.rank_offsets).numpy(), d["rank_offsets"])
    np.testing.assert_array_equal(cpu(bufs.pos).numpy(), d["pos"])
    rows = int(d["offsets"][-1])
    np.testing.assert_array_equal(cpu(bufs.row_src).numpy()[:rows], d["row_src"])
    nd = d["n_dropped"]
    assert int(cpu(bufs.n_dropped)[0]) == nd
    np.testing.assert_array_equal(cpu(bufs.drop_list).numpy()[:nd], d["drop_list"])
    # dispatched rows are exact copies of x[row_src // k]
    src_tok = torch.from_numpy(d["row_src"] // w.slots).to(bufs.xperm.device)
    assert torch.equal(bufs.xperm[:rows], inp["x"][src_tok]), "dispatched rows are not exact copies of x"
    return d


def check_ffn(w, inp, bufs, rows: int, expert_subset=None) -> float:
    """Expert outputs of the GPU's dispatched rows against the oracle's experts."""
    offs = cpu(bufs.offsets).numpy()
    fn = expert_fn(w.expert, inp["W13"], inp["W2"], w.F)
    experts = range(w.n_experts) if expert_subset is None else expert_subset
    worst = 0.0
    for e in experts:
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        X = f64(bufs.xperm[lo:hi])
        exact = fn(e, X)
        worst = max(worst, check_close(bufs.out[lo:hi], exact, bufs.out_act, f"expert {e} output",
                                       tol=TOL[w.act]))
    return worst


def check_combine(w, bufs) -> float:
    """Combine stage on the GPU's own expert outputs, gates and positions."""
    exact = orc.combine(f64(bufs.topk_gate), cpu(bufs.pos).numpy().astype(np.int64), f64(bufs.out), w.T, w.slots)
    return check_close(bufs.y, exact, w.act, "combine", tol=1e-5)


def run_layer(cfg, inp, w, device="cuda"):
    ws = abi.workspace(cfg, device)
    y = torch.full((w.T, w.d), float("nan"), dtype=w.torch_act, device=device)
    abi.moe_layer_forward(cfg, inp["x"], inp["Wg"], inp.get("bias"), inp.get("W13"), inp.get("W2"), y, ws)
    view = abi.moe_workspace_get_view(cfg, ws)
    flags = abi.moe_read_status(view.status)
    return y, ws, view, flags
