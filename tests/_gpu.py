"""GPU-side test glue: runs the library through its C ABI and compares with the oracle.

Tolerances (floating point):
  * layer output y and expert outputs: max |gpu - exact| <= tol * rms(exact), tol =
    2e-2 (bf16) or 1e-4 (fp32), as stated for the layer, with nothing added.
  * where no bf16 output can meet that bound, because the correctly rounded bf16 value
    of the exact y is already more than tol * rms(exact) away from it somewhere (a
    capacity that drops most of a hot expert's assignments shrinks rms(y) while the
    largest surviving elements keep their size): the bound is tol * rms(exact) + half
    an ulp of bf16 at the exact value, the format's own representation error on top of
    the arithmetic's budget. The Zipf workload and its gate/padded variant are such
    layers (ROUNDING_LIMITED, asserted); any other layer takes the half-ulp term only
    when its own exact output shows the same.
  * the combine stage alone (random rows and gates): tol = 1e-5 plus the half ulp of
    y's one rounding, which checks that the sum is taken in fp32 and rounded once.
  * gates: |gpu - exact| <= 2e-6 (fp32 logits carry ~1e-7 absolute error from a
    d-long dot product summed in short pieces; exp and the division add a few ulp).
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

# Workloads whose correctly rounded bf16 output alone is more than 2e-2 * rms(y) away
# from the exact y (capacity factor 1.25 with a Zipf(1.2)-skewed router: the hot expert
# drops about 95% of its assignments): the Zipf workload and its gate-policy /
# padded-layout variant, at full and reduced size.
ROUNDING_LIMITED = {"zipf_cf125", "zipf_gate_padded"}


def half_ulp(v: np.ndarray, act: str) -> np.ndarray:
    """Half an ulp of the activation dtype at |v| (bf16: 8 significant bits, fp32: 24)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-38)))
    bits = 8 if act == "bf16" else 24
    return 2.0 ** (e - bits)


def rms(v) -> float:
    v = np.asarray(v, np.float64)
    return float(np.sqrt(np.mean(v * v))) if v.size else 0.0


def output_rounding(exact, act: str) -> float:
    """max |round_act(exact) - exact| / rms(exact): how far the correctly rounded
    ``act`` value of the exact result is from it."""
    exact = np.asarray(exact, np.float64)
    if act == "f32":
        rounded = exact.astype(np.float32).astype(np.float64)
    else:
        rounded = torch.from_numpy(exact).to(torch.bfloat16).to(torch.float64).numpy()
    r = rms(exact)
    return float(np.abs(rounded - exact).max() / r) if r > 0 else 0.0


def rounding_limited(exact, act: str, tol: float) -> bool:
    """Whether no result delivered in ``act`` can be within tol * rms(exact) of the exact
    values: their own correct rounding is already farther than that somewhere."""
    return output_rounding(exact, act) > tol


def check_close(got, exact, act: str, what: str, tol: float | None = None, extra=None,
                with_half_ulp: bool = False) -> float:
    """Asserts max|got - exact| <= tol * rms(exact) elementwise (plus a per-element
    ``extra`` bound, if given; plus half an ulp of ``act`` at the exact value with
    ``with_half_ulp``, for the rounding-limited workloads and the combine-stage check);
    returns the raw max|err| / rms(exact)."""
    tol = TOL[act] if tol is None else tol
    got = f64(got)
    exact = np.asarray(exact, np.float64)
    assert got.shape == exact.shape, (what, got.shape, exact.shape)
    r = rms(exact)
    err = np.abs(got - exact)
    bound = tol * r + (half_ulp(exact, act) if with_half_ulp else np.zeros_like(exact)) + \
        (0.0 if extra is None else np.asarray(extra, np.float64))
    bad = err > bound
    assert not np.isnan(got).any(), f"{what}: NaN in GPU output"
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} elements beyond {tol}*rms{' + half-ulp' if with_half_ulp else ''}"
                             f"; worst at {i}: gpu={got[i]!r} exact={exact[i]!r} err={err[i]:.3e} "
                             f"bound={bound[i]:.3e} rms={r:.3e}")
    return float(err.max() / r) if r > 0 else 0.0


def check_layer_close(name: str, got, exact, act: str, what: str, extra=None, whole: bool = True) -> float:
    """The layer tolerance for workload ``name``: the literal bound, or, where no output
    in the activation dtype can meet it (any layer whose exact output shows it; for the
    ROUNDING_LIMITED workloads this is asserted when ``whole`` output is compared, not on
    a token sample, whose own tail may be lighter), the bound plus the output half-ulp."""
    limited = rounding_limited(exact, act, TOL[act])
    if name in ROUNDING_LIMITED and whole:
        assert limited, f"{name} is listed as rounding-limited but is not"
    return check_close(got, exact, act, what, extra=extra, with_half_ulp=limited)


class StageBuffers:
    """Output buffers of the four stage entry points, filled with sentinels. The
    dispatched-row buffers have moe_rows_capacity(cfg) rows (N*C in the padded
    layout, T*K otherwise)."""

    def __init__(self, w, cfg, device="cuda"):
        A = w.T * w.slots
        N = w.n_experts
        R = abi.moe_rows_capacity(cfg)
        i32 = dict(dtype=torch.int32, device=device)
        self.cfg, self.rows = cfg, R
        self.topk_idx = torch.full((w.T, w.slots), -7, **i32)
        self.topk_gate = torch.full((w.T, w.slots), float("nan"), dtype=torch.float32, device=device)
        self.counts_routed = torch.full((N,), -7, **i32)
        self.counts_kept = torch.full((N,), -7, **i32)
        self.offsets = torch.full((N + 1,), -7, **i32)
        self.rank_offsets = torch.full((w.D + 1,), -7, **i32)
        self.pos = torch.full((A,), -7, **i32)
        self.row_src = torch.full((max(A, R),), -7, **i32)
        self.drop_list = torch.full((A,), -7, **i32)
        self.n_dropped = torch.full((1,), -7, **i32)
        self.xperm = torch.full((R, w.d), float("nan"), dtype=w.torch_act, device=device)
        self.h = torch.full((R, max(abi.hidden_cols(cfg), 1)), float("nan"), dtype=w.torch_act, device=device)
        self.out = torch.full((R, w.d), float("nan"), dtype=abi.out_dtype(cfg), device=device)
        self.out_act = "f32" if abi.out_dtype(cfg) == torch.float32 else "bf16"
        self.y = torch.full((w.T, w.d), float("nan"), dtype=w.torch_act, device=device)
        nr = abi.moe_route_workspace_bytes(cfg)
        self.ws_route = torch.zeros(nr, dtype=torch.uint8, device=device) if nr else None
        self.ws_dispatch = torch.zeros(abi.moe_dispatch_workspace_bytes(cfg), dtype=torch.uint8, device=device)
        self.ws_ffn = torch.zeros(abi.moe_ffn_workspace_bytes(cfg), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        if w.dispatch_dtype == "fp8":
            self.xq = torch.full((R, w.d), 0xAB, dtype=torch.uint8, device=device)
            self.xscale = torch.full((R, (w.d + 127) // 128), float("nan"), dtype=torch.float32, device=device)
        if w.dispatch_dtype == "fp8_gemm":
            self.xq = torch.full((R, w.d), 0xAB, dtype=torch.uint8, device=device)
            self.xscale = torch.full((R,), float("nan"), dtype=torch.float32, device=device)
        if w.dedup:
            TD = w.T * w.D
            self.send_counts = torch.full((w.D,), -7, **i32)
            self.send_offsets = torch.full((w.D + 1,), -7, **i32)
            self.send_pos = torch.full((TD,), -7, **i32)
            self.send_src = torch.full((TD,), -7, **i32)
            if w.dispatch_dtype == "fp8":  # the send rows travel as e4m3 codes + block scales
                self.xsend = torch.full((TD, w.d), 0xAB, dtype=torch.uint8, device=device)
                self.xsend_scale = torch.full((TD, (w.d + 127) // 128), float("nan"), dtype=torch.float32,
                                              device=device)
            elif w.dispatch_dtype == "fp8_gemm":  # e4m3 codes + one scale per send row
                self.xsend = torch.full((TD, w.d), 0xAB, dtype=torch.uint8, device=device)
                self.xsend_scale = torch.full((TD,), float("nan"), dtype=torch.float32, device=device)
            else:
                self.xsend = torch.full((TD, w.d), float("nan"), dtype=w.torch_act, device=device)

    def smap(self):
        return abi.send_map(self.send_counts, self.send_offsets, self.send_pos, self.send_src)

    def dedup(self, inp, topk_idx, pos, xperm, xq=None, xscale=None):
        """The deduplicated dispatch into xperm, or (FP8 GEMM format) into xq / xscale."""
        if self.cfg.dispatch_dtype == abi.MOE_DISPATCH_FP8_GEMM:
            abi.moe_dispatch_dedup_fp8_gemm(self.cfg, inp["x"], topk_idx, pos, self.smap(), self.xsend,
                                            self.xsend_scale, xq, xscale, self.ws_dispatch)
            return
        if self.cfg.dispatch_dtype == abi.MOE_DISPATCH_FP8:
            abi.moe_dispatch_dedup_fp8(self.cfg, inp["x"], topk_idx, pos, self.smap(), self.xsend, self.xsend_scale,
                                       xperm, self.ws_dispatch)
            return
        abi.moe_dispatch_dedup(self.cfg, inp["x"], topk_idx, pos, self.smap(), self.xsend, xperm, self.ws_dispatch)

    def dmap(self):
        return abi.dispatch_map(self.counts_routed, self.counts_kept, self.offsets, self.rank_offsets, self.pos,
                                self.row_src, self.drop_list, self.n_dropped)

    def route(self, inp):
        abi.moe_route(self.cfg, inp["x"], inp["Wg"], inp.get("bias"), self.topk_idx, self.topk_gate, self.ws_route)

    def dispatch(self, inp, topk_idx=None, topk_gate=None):
        abi.moe_dispatch(self.cfg, inp["x"], self.topk_idx if topk_idx is None else topk_idx, self.dmap(),
                         self.xperm, self.ws_dispatch, topk_gate=self.topk_gate if topk_gate is None else topk_gate)

    def ffn(self, inp, xperm=None, offsets=None, xq=None, xscale=None):
        offsets = self.offsets if offsets is None else offsets
        if self.cfg.dispatch_dtype == abi.MOE_DISPATCH_FP8_GEMM:
            abi.moe_expert_ffn_fp8(self.cfg, self.xq if xq is None else xq, self.xscale if xscale is None else xscale,
                                   offsets, api_w13(self.cfg, inp), api_w2(self.cfg, inp), self.h, self.out,
                                   self.ws_ffn)
            return
        abi.moe_expert_ffn(self.cfg, self.xperm if xperm is None else xperm, offsets, inp["W13"], inp["W2"],
                           self.h, self.out, self.ws_ffn)

    def combine(self, out=None, topk_gate=None, pos=None):
        abi.moe_combine(self.cfg, self.out if out is None else out, self.topk_gate if topk_gate is None else topk_gate,
                        self.pos if pos is None else pos, self.y, self.status)

    def dispatch_status(self) -> int:
        return abi.moe_read_status(self.ws_dispatch.data_ptr())

    def ffn_status(self) -> int:
        return abi.moe_read_status(self.ws_ffn.data_ptr())


def api_w13(cfg, inp):
    """The W13 the library takes for this config: the bf16 weights, or (FP8 GEMM) their
    FP8 buffer, quantized once on the device by the library and kept in ``inp``."""
    if cfg.dispatch_dtype != abi.MOE_DISPATCH_FP8_GEMM or inp.get("W13") is None:
        return inp.get("W13")
    if "W13_fp8" not in inp:
        inp["W13_fp8"] = abi.fp8_weights(cfg, inp["W13"])
    return inp["W13_fp8"]


def api_w2(cfg, inp):
    """The W2 the library takes: the bf16 weights, or (FP8 hidden activation) their FP8
    buffer, quantized once on the device by the library and kept in ``inp``."""
    if cfg.precision != abi.MOE_PRECISION_FP8_H or inp.get("W2") is None:
        return inp.get("W2")
    if "W2_fp8" not in inp:
        inp["W2_fp8"] = abi.fp8_w2(cfg, inp["W2"])
    return inp["W2_fp8"]


# Relative error of the GPU's fp32 hidden activation against the exact one that the FP8
# hidden-activation budget allows for: fp32 sums of K exact e4m3 products and the fast
# exp/divide of silu stay near 1e-6; 2^-16 leaves a margin.
FP8_H_EPS = 2.0 ** -16


def fp8_h_jump(h, eps: float = FP8_H_EPS) -> np.ndarray:
    """How far the FP8 form of each element of h (``fp8_hidden``, a step function of h)
    can move when h is off by a relative eps: the e4m3 code the GPU picks from its own
    bf16 h may differ from the oracle's next to a rounding boundary, as a top-k may
    differ at a near tie."""
    mid = orc.fp8_hidden(h)
    return np.maximum(np.abs(orc.fp8_hidden(h * (1 - eps)) - mid), np.abs(orc.fp8_hidden(h * (1 + eps)) - mid))


def fp8_h_budget(w, inp, e, X) -> np.ndarray:
    """Bound [rows, d] on what those code changes can move expert e's outputs for the
    rows X: sum over features of the jump times |W2| (row-quantized). The quantized
    weights are kept in ``inp`` after first use."""
    cache = inp.setdefault("_fp8_h_budget_cache", {})
    if e not in cache:
        shared = inp.get("_expert_cache", {})  # the expert function's quantized weights, if it ran first
        if e in shared:
            w13q, w2q = shared[e]
        else:
            w13q = orc.quantize_fp8_rows(f64(inp["W13"][e]))["deq"]
            w2q = orc.quantize_fp8_rows(f64(inp["W2"][e]))["deq"]  # [d, F]
        cache[e] = (w13q, np.abs(w2q).T.astype(np.float32))
    w13q, w2abs = cache[e]
    X = np.asarray(X, np.float64)
    F = w.F
    h = orc.hidden_relu(X, w13q.T) if w.expert == "relu" else orc.hidden_swiglu(X, w13q[:F].T, w13q[F:].T)
    return (fp8_h_jump(h).astype(np.float32) @ w2abs).astype(np.float64)


def fp8_h_layer_budget(w, inp, ref) -> np.ndarray:
    """The same bound carried through the combine: [T, d] for an oracle forward ``ref``."""
    out_b = np.zeros_like(ref["out"])
    off = ref["offsets"]
    for e in range(w.n_experts):
        lo, hi = int(off[e]), int(off[e + 1])
        held = np.arange(lo, hi)[ref["row_src"][lo:hi] >= 0]
        if held.size:
            out_b[held] = fp8_h_budget(w, inp, e, ref["xperm"][held])
    return orc.combine(ref["G"], ref["pos"], out_b, w.T, w.slots)


def check_fp8_weights(w, cfg, inp, experts) -> None:
    """The library's FP8 weight buffer: codes and per-row scales of the given experts
    bit-exact against the oracle's row-wise quantization of W13."""
    codes, scales = abi.fp8_weight_parts(cfg, api_w13(cfg, inp), w.n_experts, w.w13_rows, w.d)
    for e in experts:
        q = orc.quantize_fp8_rows(f64(inp["W13"][e]))
        np.testing.assert_array_equal(cpu(codes[e]).numpy(), q["codes"])
        np.testing.assert_array_equal(cpu(scales[e]).numpy().astype(np.float64), q["scales"])
    if cfg.precision == abi.MOE_PRECISION_FP8_H:  # the W2 buffer has the same layout: [N, d, F] + [N, d]
        codes, scales = abi.fp8_weight_parts(cfg, api_w2(cfg, inp), w.n_experts, w.d, w.F)
        for e in experts:
            q = orc.quantize_fp8_rows(f64(inp["W2"][e]))
            np.testing.assert_array_equal(cpu(codes[e]).numpy(), q["codes"])
            np.testing.assert_array_equal(cpu(scales[e]).numpy().astype(np.float64), q["scales"])


def compare_fp8_rows(w, xq, xscale, row_src, x, rows=None) -> int:
    """FP8-GEMM dispatch: the codes and row scale of every kept row (or of ``rows``)
    bit-exact against the oracle's row-wise quantization of its token's row."""
    rs = np.asarray(row_src)
    held = np.nonzero(rs >= 0)[0] if rows is None else np.asarray(rows)
    tok = rs[held] // w.slots
    q = orc.quantize_fp8_rows(f64(x[torch.from_numpy(tok).to(x.device)]))
    np.testing.assert_array_equal(cpu(xq).numpy()[held], q["codes"])
    np.testing.assert_array_equal(cpu(xscale).numpy().astype(np.float64)[held], q["scales"])
    return int(held.size)


def cpu(t):
    return t.detach().cpu()


def capacity_of(cfg):
    return None if cfg.capacity < 0 else int(cfg.capacity)


def oracle_route(w, inp) -> dict:
    """The oracle's router on the original inputs, with the shared slots appended.
    Under a group limit the near ties are those of the group choice and those of
    KeepTopK inside the kept groups."""
    H = orc.router_logits(f64(inp["x"]), f64(inp["Wg"]), f64(inp.get("bias")))
    Hs = selectable_logits(w, H)
    idx = orc.keep_topk(Hs, w.k)
    G = orc.kept_softmax(H, idx)
    tie = route_tie_flags(w, H)
    S = w.n_shared
    idx_full = np.concatenate([idx, np.broadcast_to(w.E + np.arange(S), (w.T, S))], axis=1)
    G_full = np.concatenate([G, np.ones((w.T, S))], axis=1)
    return dict(H=H, idx=idx, G=G, tie=tie, idx_full=idx_full, G_full=G_full)


def selectable_logits(w, H):
    """H with the logits outside each token's kept groups at -inf (group-limited routing)."""
    if 0 < w.topk_groups < w.n_groups:
        return np.where(orc.group_allowed(H, w.n_groups, w.topk_groups), H, -np.inf)
    return H


def route_tie_flags(w, H):
    """Near ties of the selection: KeepTopK's (inside the kept groups) and the group choice's."""
    s, o = orc.near_tie_flags(selectable_logits(w, H), w.k)
    tie = s | o
    if 0 < w.topk_groups < w.n_groups:
        tie |= orc.group_tie_flags(H, w.n_groups, w.topk_groups)
    return tie


def check_route(w, inp, bufs, ref=None) -> dict:
    """Top-k ids exact away from near ties; gates within GATE_TOL. Returns stats."""
    ref = oracle_route(w, inp) if ref is None else ref
    idx_o, G_o, tie = ref["idx"], ref["G"], ref["tie"]
    idx_all = cpu(bufs.topk_idx).numpy()
    G_all = cpu(bufs.topk_gate).numpy().astype(np.float64)
    S = w.n_shared
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
    return dict(ref, near_ties=int(tie.sum()), flipped=int(mismatch.sum()), gate_err=float(gerr))


def gate_boundary_ties(w, idx, G, capacity, tol=2 * GATE_TOL) -> np.ndarray:
    """Tokens whose gate on a capped, overflowing expert lies within ``tol`` of that
    expert's keep cutoff (the capacity-th largest gate): under the gate drop policy
    an fp32 and an fp64 router may keep different ones of them."""
    flag = np.zeros(w.T, bool)
    if capacity is None:
        return flag
    for e in range(w.E):
        tok, slot = np.nonzero(idx == e)
        if tok.size <= capacity:
            continue
        g = G[tok, slot]
        order = np.sort(g)[::-1]
        cut = order[capacity - 1] if capacity > 0 else np.inf
        flag[tok[np.abs(g - cut) <= tol]] = True
        if capacity > 0:
            nxt = order[capacity]
            flag[tok[np.abs(g - nxt) <= tol]] = True
    return flag


def compare_dispatch(w, bufs, d, x=None, xperm=None, fp8_rows=None):
    """Every routing-map array bit-exact against the oracle's dispatch ``d``; the
    dispatched rows exact copies of x (padding rows zero)."""
    np.testing.assert_array_equal(cpu(bufs.counts_routed).numpy(), d["counts_routed"])
    np.testing.assert_array_equal(cpu(bufs.counts_kept).numpy(), d["counts_kept"])
    np.testing.assert_array_equal(cpu(bufs.offsets).numpy(), d["offsets"])
    np.testing.assert_array_equal(cpu(bufs.rank_offsets).numpy(), d["rank_offsets"])
    np.testing.assert_array_equal(cpu(bufs.pos).numpy(), d["pos"])
    rows = d["row_src"].size
    np.testing.assert_array_equal(cpu(bufs.row_src).numpy()[:rows], d["row_src"])
    nd = d["n_dropped"]
    assert int(cpu(bufs.n_dropped)[0]) == nd
    np.testing.assert_array_equal(cpu(bufs.drop_list).numpy()[:nd], d["drop_list"])
    if x is not None:
        xperm = bufs.xperm if xperm is None else xperm
        src = torch.from_numpy(d["row_src"]).to(xperm.device)
        valid = src >= 0
        expect = x[src[valid] // w.slots]
        if fp8_rows is not None:  # the FP8 dispatch's routed rows are the dequantized rows of x
            q = torch.from_numpy(orc.quantize_fp8_blocks(f64(expect))["deq"]).to(expect.dtype).to(expect.device)
            routed = (torch.from_numpy(np.asarray(fp8_rows)).to(xperm.device))[valid]
            expect = torch.where(routed[:, None], q, expect)
        assert torch.equal(xperm[:rows][valid], expect), "dispatched rows are not exact copies of x"
        assert torch.count_nonzero(xperm[:rows][~valid]) == 0, "padding rows are not zero"


def oracle_dispatch(w, idx, gates, capacity):
    return orc.dispatch(np.asarray(idx, np.int64), w.n_experts, capacity, w.D, capped_experts=w.E,
                        gates=None if gates is None else np.asarray(gates, np.float64),
                        drop_policy=w.drop_policy, layout=w.layout)


def check_dispatch_of_oracle_routing(w, inp, cfg, r, capacity) -> dict:
    """The GPU dispatch run on the oracle's own routing (its top-k ids, and its gates
    rounded to fp32 for the gate drop policy) against the oracle's dispatch of the same
    ids and gates: every map array and every row bit for bit, at any size and whatever
    near ties the GPU's router met. The inputs go from the oracle to the GPU, never the
    other way."""
    b = StageBuffers(w, cfg)
    idx = torch.from_numpy(np.ascontiguousarray(r["idx_full"]).astype(np.int32)).cuda()
    gates32 = np.ascontiguousarray(r["G_full"]).astype(np.float32)
    b.dispatch(inp, topk_idx=idx, topk_gate=torch.from_numpy(gates32).cuda())
    d = oracle_dispatch(w, r["idx_full"], gates32.astype(np.float64), capacity)
    torch.cuda.synchronize()
    assert b.dispatch_status() == 0
    if w.dispatch_dtype == "fp8_gemm":  # the dispatched rows themselves are checked as e4m3 codes elsewhere
        compare_dispatch(w, b, d)
    else:
        compare_dispatch(w, b, d, inp["x"])
    return d


def check_near_tie_count(w, ws, view, H) -> int:
    """The forward's own near-tie count (tokens whose k-th and (k+1)-th largest fp32
    logits are within 1e-6 relative) against the oracle's float64 logits: it must lie
    between the number of tokens with a float64 gap below 0.5e-6 and below 2e-6 (fp32
    logits are off by about 1e-7 absolute, which moves a gap by far less than that
    band near the selected logits' magnitudes). Returns the GPU count."""
    base = ws.data_ptr()
    n = int(ws[view.n_near_ties - base:view.n_near_ties - base + 4].view(torch.int32).cpu()[0])
    Hs = selectable_logits(w, H)
    lo = int(orc.near_tie_flags(Hs, w.k, rel=0.5e-6)[0].sum())
    hi = int(orc.near_tie_flags(Hs, w.k, rel=2e-6)[0].sum())
    assert lo <= n <= hi, f"near-tie count {n} outside [{lo}, {hi}]"
    return n


def check_dispatch(w, inp, bufs, capacity, st) -> dict:
    """Dispatch stage on seeded synthetic ids and gates (``st`` from
    workloads.make_stage_inputs): every map array bit-exact, rows copied exactly."""
    bufs.dispatch(inp, topk_idx=st["topk_idx"], topk_gate=st["topk_gate"])
    d = oracle_dispatch(w, cpu(st["topk_idx"]).numpy(), cpu(st["topk_gate"]).numpy(), capacity)
    torch.cuda.synchronize()
    compare_dispatch(w, bufs, d, inp["x"])
    return d


def check_dedup(w, inp, bufs, st, d) -> dict:
    """Deduplicated dispatch on the synthetic ids' dispatch map ``d`` (already on the
    GPU in ``bufs``): the send map bit-exact against the oracle, the send rows exact
    copies of x (FP8: their codes and block scales bit-exact against the oracle's
    quantization of x), and the fanned-out expert rows equal to the direct gather's
    (FP8: to the direct FP8 dispatch's dequantized rows)."""
    fp8 = w.dispatch_dtype == "fp8"
    if w.dispatch_dtype == "fp8_gemm":
        return check_dedup_fp8_gemm(w, inp, bufs, st, d)
    direct = bufs.xperm.clone()
    if fp8:  # the direct FP8 dispatch of the same map: routed rows dequantized, shared rows from x
        direct = torch.full_like(bufs.xperm, float("nan"))
        xq = torch.empty(bufs.rows, w.d, dtype=torch.uint8, device=direct.device)
        xs = torch.empty(bufs.rows, (w.d + 127) // 128, dtype=torch.float32, device=direct.device)
        abi.moe_dispatch_fp8(bufs.cfg, inp["x"], st["topk_idx"], bufs.dmap(), xq, xs, direct, bufs.ws_dispatch)
    fanned = torch.full_like(bufs.xperm, float("nan"))
    bufs.dedup(inp, st["topk_idx"], bufs.pos, fanned)
    s = orc.dedup_send(cpu(st["topk_idx"]).numpy(), d["pos"], w.E, w.D)
    torch.cuda.synchronize()
    assert bufs.dispatch_status() == 0
    np.testing.assert_array_equal(cpu(bufs.send_counts).numpy(), s["send_counts"])
    np.testing.assert_array_equal(cpu(bufs.send_offsets).numpy(), s["send_offsets"])
    np.testing.assert_array_equal(cpu(bufs.send_pos).numpy(), s["send_pos"])
    n = s["n_send"]
    np.testing.assert_array_equal(cpu(bufs.send_src).numpy()[:n], s["send_src"])
    src_tok = torch.from_numpy(s["send_src"] // w.D).to(bufs.xsend.device)
    if fp8:
        q = orc.quantize_fp8_blocks(f64(inp["x"][src_tok]))
        np.testing.assert_array_equal(cpu(bufs.xsend).numpy()[:n], q["codes"])
        np.testing.assert_array_equal(cpu(bufs.xsend_scale).numpy().astype(np.float64)[:n], q["scales"])
    else:
        assert torch.equal(bufs.xsend[:n], inp["x"][src_tok]), "send rows are not exact copies of x"
    held = torch.from_numpy(np.nonzero(d["row_src"] >= 0)[0]).to(fanned.device)  # padding rows are not sent
    assert torch.equal(fanned[held], direct[held]), "fanned-out rows differ from the direct dispatch's"
    return s


def check_dedup_fp8_gemm(w, inp, bufs, st, d) -> dict:
    """Deduplicated dispatch in the FP8 GEMM's format: the send map bit-exact against the
    oracle, each send row's codes and scale bit-exact against the oracle's row quantization
    of its token, and the expert rows' codes and scales the fan-out writes equal to the
    direct FP8 dispatch's of the same map (and so to the oracle's)."""
    R = bufs.rows
    dq = torch.full((R, w.d), 0xAB, dtype=torch.uint8, device=bufs.xq.device)
    ds = torch.full((R,), float("nan"), dtype=torch.float32, device=bufs.xq.device)
    abi.moe_dispatch_fp8(bufs.cfg, inp["x"], st["topk_idx"], bufs.dmap(), dq, ds, None, bufs.ws_dispatch)
    fq = torch.full_like(dq, 0xCD)
    fs = torch.full_like(ds, float("nan"))
    bufs.dedup(inp, st["topk_idx"], bufs.pos, None, xq=fq, xscale=fs)
    s = orc.dedup_send(cpu(st["topk_idx"]).numpy(), d["pos"], w.E, w.D)
    torch.cuda.synchronize()
    assert bufs.dispatch_status() == 0
    np.testing.assert_array_equal(cpu(bufs.send_counts).numpy(), s["send_counts"])
    np.testing.assert_array_equal(cpu(bufs.send_offsets).numpy(), s["send_offsets"])
    np.testing.assert_array_equal(cpu(bufs.send_pos).numpy(), s["send_pos"])
    n = s["n_send"]
    np.testing.assert_array_equal(cpu(bufs.send_src).numpy()[:n], s["send_src"])
    q = orc.quantize_fp8_rows(f64(inp["x"][torch.from_numpy(s["send_src"] // w.D).to(inp["x"].device)]))
    np.testing.assert_array_equal(cpu(bufs.xsend).numpy()[:n], q["codes"])
    np.testing.assert_array_equal(cpu(bufs.xsend_scale).numpy().astype(np.float64)[:n], q["scales"])
    held = torch.from_numpy(np.nonzero(d["row_src"] >= 0)[0]).to(fq.device)
    assert torch.equal(fq[held], dq[held]), "fanned-out codes differ from the direct FP8 dispatch's"
    assert torch.equal(fs[held], ds[held]), "fanned-out row scales differ from the direct FP8 dispatch's"
    compare_fp8_rows(w, fq, fs, d["row_src"], inp["x"])
    return s


def check_fp8(w, inp, bufs, st, d) -> dict:
    """FP8 dispatch of the synthetic ids' dispatch map ``d``: every routed row's e4m3
    codes and block scales bit-exact against the oracle's quantization of its token,
    the receiving side's bf16 rows equal to the oracle's dequantized values, shared
    experts' rows equal to x. FP8 GEMM format: every kept row's codes and row scale."""
    if w.dispatch_dtype == "fp8_gemm":
        abi.moe_dispatch_fp8(bufs.cfg, inp["x"], st["topk_idx"], bufs.dmap(), bufs.xq, bufs.xscale, None,
                             bufs.ws_dispatch)
        torch.cuda.synchronize()
        assert bufs.dispatch_status() == 0
        return dict(rows=compare_fp8_rows(w, bufs.xq, bufs.xscale, d["row_src"], inp["x"]))
    rows_out = torch.full_like(bufs.xperm, float("nan"))
    abi.moe_dispatch_fp8(bufs.cfg, inp["x"], st["topk_idx"], bufs.dmap(), bufs.xq, bufs.xscale, rows_out,
                         bufs.ws_dispatch)
    q = orc.quantize_fp8_blocks(f64(inp["x"]))
    torch.cuda.synchronize()
    assert bufs.dispatch_status() == 0
    idx = cpu(st["topk_idx"]).numpy().reshape(-1)
    rs = d["row_src"]
    rows = np.nonzero(rs >= 0)[0]
    routed = rows[idx[rs[rows]] < w.E]
    shared = rows[idx[rs[rows]] >= w.E]
    tok = rs[routed] // w.slots
    np.testing.assert_array_equal(cpu(bufs.xq).numpy()[routed], q["codes"][tok])
    np.testing.assert_array_equal(cpu(bufs.xscale).numpy().astype(np.float64)[routed], q["scales"][tok])
    got = f64(rows_out)
    np.testing.assert_array_equal(got[routed], q["deq"][tok])
    if shared.size:
        np.testing.assert_array_equal(got[shared], f64(inp["x"])[rs[shared] // w.slots])
    return dict(rows=int(routed.size), mean_abs_scale_exp=float(np.abs(q["exps"]).mean()))


def check_ffn(w, inp, bufs, st, expert_subset=None) -> float:
    """Expert FFN stage on seeded synthetic rows and per-expert counts: each
    expert's output rows against the oracle's expert on the same rows."""
    counts = st["counts"].numpy()
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    fp8 = w.dispatch_dtype == "fp8_gemm"
    rows_in = f64(st["xperm"])
    if fp8:  # the FP8 GEMM's input rows: the oracle's row-wise quantization of the synthetic rows
        q = orc.quantize_fp8_rows(rows_in)
        rows_in = q["deq"]
        xq = torch.zeros(bufs.rows, w.d, dtype=torch.uint8, device="cuda")
        xq[:offs[-1]] = torch.from_numpy(q["codes"]).cuda()
        xs = torch.zeros(bufs.rows, dtype=torch.float32, device="cuda")
        xs[:offs[-1]] = torch.from_numpy(q["scales"]).float().cuda()
        bufs.ffn(inp, offsets=torch.from_numpy(offs).cuda(), xq=xq, xscale=xs)
    else:
        xperm = torch.zeros(bufs.rows, w.d, dtype=w.torch_act, device="cuda")
        xperm[:offs[-1]] = st["xperm"]
        bufs.ffn(inp, xperm=xperm, offsets=torch.from_numpy(offs).cuda())
    fn = expert_fn(w.expert, inp["W13"], inp["W2"], w.F, fp8_up=fp8, fp8_h=w.precision == "fp8_h")
    experts = range(w.n_experts) if expert_subset is None else expert_subset
    if fp8:
        check_fp8_weights(w, bufs.cfg, inp, [e for e in experts if counts[e] > 0][:3])
    worst = 0.0
    for e in experts:
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        exact = fn(e, rows_in[lo:hi])
        if w.precision == "fp8_h":
            worst = max(worst, check_close(bufs.out[lo:hi], exact, bufs.out_act, f"expert {e} output",
                                           tol=TOL[w.act], extra=fp8_h_budget(w, inp, e, rows_in[lo:hi])))
            continue
        worst = max(worst, check_close(bufs.out[lo:hi], exact, bufs.out_act, f"expert {e} output",
                                       tol=TOL[w.act]))
    return worst


def check_combine(w, bufs, st) -> float:
    """Combine stage on seeded synthetic expert rows, gates and positions."""
    out = st["out_rows"].to(bufs.out.dtype)
    if out.shape[0] < bufs.rows:
        out = torch.cat([out, torch.zeros(bufs.rows - out.shape[0], w.d, dtype=out.dtype, device=out.device)])
    bufs.combine(out=out, topk_gate=st["topk_gate"], pos=st["pos"])
    exact = orc.combine(f64(st["topk_gate"]), cpu(st["pos"]).numpy().astype(np.int64), f64(out), w.T, w.slots)
    return check_close(bufs.y, exact, w.act, "combine", tol=1e-5, with_half_ulp=True)


def check_map_properties(w, m, capacity):
    """What any correct dispatch of the GPU's own ids satisfies, at any size: counts
    are the ids' histogram, offsets their prefix sum (or e*C), each kept assignment's
    row lies in its expert's segment, row_src inverts pos, rows inside a segment are
    in token order, nothing is kept beyond the capacity."""
    idx = cpu(m.topk_idx).numpy().astype(np.int64)
    N, A = w.n_experts, w.T * w.slots
    flat = idx.reshape(-1)
    routed = np.bincount(flat, minlength=N)
    np.testing.assert_array_equal(cpu(m.counts_routed).numpy(), routed)
    kept = cpu(m.counts_kept).numpy().astype(np.int64)
    capped = np.arange(N) < w.E
    limit = np.where(capped & (capacity is not None), capacity if capacity is not None else 0, routed)
    np.testing.assert_array_equal(kept, np.minimum(routed, limit))
    offs = cpu(m.offsets).numpy().astype(np.int64)
    if w.layout == "padded":
        np.testing.assert_array_equal(offs, np.arange(N + 1) * capacity)
    else:
        np.testing.assert_array_equal(offs, np.concatenate([[0], np.cumsum(kept)]))
    pos = cpu(m.pos).numpy().astype(np.int64)
    row_src = cpu(m.row_src).numpy().astype(np.int64)
    k_mask = pos >= 0
    assert k_mask.sum() == kept.sum() and int(cpu(m.n_dropped)[0]) == A - kept.sum()
    a = np.nonzero(k_mask)[0]
    e = flat[a]
    assert np.all((pos[a] >= offs[e]) & (pos[a] < offs[e] + kept[e]))
    np.testing.assert_array_equal(row_src[pos[a]], a)
    for ee in range(N):
        seg = row_src[offs[ee]:offs[ee] + kept[ee]]
        assert np.all(np.diff(seg) > 0), f"expert {ee}: rows not in token order"


def check_chained_dispatch(w, inp, m, r, capacity, xperm=None) -> str:
    """The GPU's dispatch of its own routing. Where its ids equal the oracle's (no
    near-tie flip) and, under the gate drop policy, no two gates meet at a keep
    cutoff, it must equal the oracle's dispatch of the oracle's routing bit for bit;
    otherwise it is held to the properties every correct dispatch has."""
    exact = r["flipped"] == 0
    if exact and w.drop_policy == "gate":
        exact = not gate_boundary_ties(w, r["idx"], r["G"], capacity).any()
    if exact:
        d = oracle_dispatch(w, r["idx_full"], r["G_full"], capacity)
        if w.dispatch_dtype == "fp8_gemm":  # rows travel only as codes + row scales
            compare_dispatch(w, m, d)
            if xperm is None:
                sample = np.nonzero(d["row_src"] >= 0)[0]
                sample = np.random.default_rng(2).choice(sample, size=min(256, sample.size), replace=False)
                compare_fp8_rows(w, m.xq, m.xscale, d["row_src"], inp["x"], rows=sample)
            return "exact"
        fp8_rows = None
        if w.dispatch_dtype == "fp8":  # rows holding a routed assignment travel as FP8
            rs = d["row_src"]
            fp8_rows = (rs >= 0) & (r["idx_full"].reshape(-1)[np.maximum(rs, 0)] < w.E)
        compare_dispatch(w, m, d, inp["x"], xperm, fp8_rows)
        return "exact"
    check_map_properties(w, m, capacity)
    return "properties"


class WorkspaceMap:
    """The dispatch map inside a forward's workspace, as tensors named like StageBuffers'."""

    def __init__(self, w, cfg, ws, view):
        A, N = w.T * w.slots, w.n_experts
        R = abi.moe_rows_capacity(cfg)
        base = ws.data_ptr()
        i32 = lambda ptr, n: ws[ptr - base:ptr - base + 4 * n].view(torch.int32)
        mp = view
        self.topk_idx = i32(view.topk_idx, A).view(w.T, w.slots)
        self.topk_gate = ws[view.topk_gate - base:view.topk_gate - base + 4 * A].view(torch.float32).view(w.T, w.slots)
        self.counts_routed = i32(mp.counts_routed, N)
        self.counts_kept = i32(mp.counts_kept, N)
        self.offsets = i32(mp.offsets, N + 1)
        self.rank_offsets = i32(mp.rank_offsets, w.D + 1)
        self.pos = i32(mp.pos, A)
        self.row_src = i32(mp.row_src, max(A, R))
        self.drop_list = i32(mp.drop_list, A)
        self.n_dropped = i32(mp.n_dropped, 1)
        esz = torch.tensor([], dtype=w.torch_act).element_size()
        self.xperm = ws[view.xperm - base:view.xperm - base + R * w.d * esz].view(w.torch_act).view(R, w.d)
        odt = abi.out_dtype(cfg)
        osz = torch.tensor([], dtype=odt).element_size()
        self.out = None if not view.out else \
            ws[view.out - base:view.out - base + R * w.d * osz].view(odt).view(R, w.d)
        self.out_act = "f32" if odt == torch.float32 else "bf16"
        if w.dispatch_dtype == "fp8_gemm" or (w.dispatch_dtype == "fp8" and not w.dedup):
            nb = (w.d + 127) // 128 if w.dispatch_dtype == "fp8" else 1
            self.xq = ws[view.xq - base:view.xq - base + R * w.d].view(R, w.d)
            self.xscale = ws[view.xscale - base:view.xscale - base + 4 * R * nb].view(torch.float32).view(R, nb)
            if w.dispatch_dtype == "fp8_gemm":
                self.xscale = self.xscale.view(R)
        if w.dedup:
            TD = w.T * w.D
            self.send_counts = i32(view.send_counts, w.D)
            self.send_offsets = i32(view.send_offsets, w.D + 1)
            self.send_pos = i32(view.send_pos, TD)
            self.send_src = i32(view.send_src, TD)
            if w.dispatch_dtype in ("fp8", "fp8_gemm"):  # codes [TD, d] and block or row scales of the send rows
                nb = (w.d + 127) // 128 if w.dispatch_dtype == "fp8" else 1
                self.xsend = ws[view.xsend - base:view.xsend - base + TD * w.d].view(TD, w.d)
                self.xsend_scale = ws[view.xsend_scale - base:view.xsend_scale - base + 4 * TD * nb] \
                    .view(torch.float32).view(TD, nb)
            else:
                self.xsend = ws[view.xsend - base:view.xsend - base + TD * w.d * esz].view(w.torch_act).view(TD, w.d)


def chain(w, inp, cfg) -> StageBuffers:
    """The four stage entry points chained on the GPU, each on the previous one's output."""
    b = StageBuffers(w, cfg)
    b.route(inp)
    b.dispatch(inp)
    if w.dispatch_dtype == "fp8":  # the routed rows travel as FP8 and come back as bf16
        abi.moe_dispatch_fp8(cfg, inp["x"], b.topk_idx, b.dmap(), b.xq, b.xscale, b.xperm, b.ws_dispatch)
    if w.dispatch_dtype == "fp8_gemm":  # every row travels as row-scaled FP8, read by the FP8 GEMM as it is
        abi.moe_dispatch_fp8(cfg, inp["x"], b.topk_idx, b.dmap(), b.xq, b.xscale, None, b.ws_dispatch)
    if w.expert != "identity":
        b.ffn(inp)
        b.combine()
    else:
        b.combine(out=b.xperm)
    torch.cuda.synchronize()
    return b


def run_layer(cfg, inp, w, device="cuda"):
    ws = abi.workspace(cfg, device)
    y = torch.full((w.T, w.d), float("nan"), dtype=w.torch_act, device=device)
    abi.moe_layer_forward(cfg, inp["x"], inp["Wg"], inp.get("bias"), api_w13(cfg, inp), api_w2(cfg, inp), y, ws)
    view = abi.moe_workspace_get_view(cfg, ws)
    flags = abi.moe_read_status(view.status)
    return y, ws, view, flags
