"""GPU parity: the CUDA path through the C ABI against the float64 CPU oracle.

Every oracle input comes from the seeded generators, never from the CUDA path:
the router is checked on the original inputs; dispatch, expert FFN and combine
each run on seeded synthetic inputs of their own (workloads.make_stage_inputs);
the GPU's chained dispatch is compared with the oracle's dispatch of the oracle's
routing where the two routings agree; end-to-end checks run the whole layer from
the original inputs and exclude only near-tie tokens. Reduced sizes span several
tiles and ragged tails; the full workload sizes are checked on sampled experts and
tokens in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from routing_dispatch_combine_moe_b300 import abi
from routing_dispatch_combine_moe_b300 import workloads as wl
from tests._gpu import (StageBuffers, WorkspaceMap, capacity_of, chain, check_chained_dispatch, check_close,
                        compare_fp8_rows,
                        check_dispatch_of_oracle_routing, check_layer_close, check_near_tie_count,
                        check_combine, check_dedup, check_dispatch, check_ffn, check_fp8, check_route, cpu,
                        fp8_h_budget, fp8_h_layer_budget, gate_boundary_ties, half_ulp, oracle_dispatch,
                        oracle_route, rms, route_tie_flags, run_layer)
from tests._harness import expert_fn, f64, run_oracle

pytestmark = pytest.mark.gpu

W = wl.WORKLOADS
REDUCED = {
    "tiny_f32": W["tiny_f32"],
    "mixtral_bf16": wl.scaled(W["mixtral_bf16"], T=512, d=1024, F=1536),
    "dsv3_route_only": W["dsv3_route_only"],
    "zipf_cf125": wl.scaled(W["zipf_cf125"], T=2048, d=512, F=384),
    "dsv3_full": wl.scaled(W["dsv3_full"], T=512, d=1024, F=256),
    "dsv3_decode": wl.scaled(W["dsv3_decode"], d=1024, F=256),
    "zipf_gate_padded": wl.scaled(W["zipf_cf125"], T=2048, d=512, F=384, drop_policy="gate", layout="padded"),
    "grouped_dedup": wl.scaled(W["dsv3_grouped_dedup"], T=512, d=1024),
    "grouped_dedup_swiglu": wl.Workload("grouped_dedup_swiglu", T=700, d=512, E=64, k=6, F=256, act="bf16",
                                        expert="swiglu", D=8, n_groups=8, topk_groups=3, dedup=True,
                                        capacity_factor="1"),
    # FP8 send rows with the deduplicated dispatch: identity experts with a ragged last block,
    # and SwiGLU experts with a shared expert and drops
    "grouped_dedup_fp8": wl.scaled(W["dsv3_grouped_dedup_fp8"], T=512, d=1088),
    "grouped_dedup_fp8_swiglu": wl.Workload("grouped_dedup_fp8_swiglu", T=700, d=512, E=64, k=6, F=256,
                                            act="bf16", expert="swiglu", D=8, n_groups=8, topk_groups=3, dedup=True,
                                            capacity_factor="1", n_shared=1, dispatch_dtype="fp8"),
    # row-scaled FP8 send rows handed to the FP8 GEMM: a shared expert (quantized from x on
    # the receiving side) and drops
    "grouped_dedup_fp8_gemm": wl.Workload("grouped_dedup_fp8_gemm", T=700, d=512, E=64, k=6, F=256, act="bf16",
                                          expert="swiglu", D=8, n_groups=8, topk_groups=3, dedup=True,
                                          capacity_factor="1", n_shared=1, dispatch_dtype="fp8_gemm"),
    "mixtral_fp8": wl.scaled(W["mixtral_fp8_dispatch"], T=512, d=1024, F=1536),
    "decode_fp8": wl.scaled(W["dsv3_decode"], d=1088, F=256, dispatch_dtype="fp8"),  # ragged last block
    "mixtral_fp8_gemm": wl.scaled(W["mixtral_fp8_gemm"], T=512, d=1024, F=1536),
    # shared expert, 8 virtual ranks, d not a multiple of 128 (a partial last K block)
    "decode_fp8_gemm": wl.scaled(W["dsv3_decode"], d=1072, F=256, dispatch_dtype="fp8_gemm"),
    "relu_fp8_gemm": wl.Workload("relu_fp8_gemm", T=300, d=512, E=6, k=2, F=448, act="bf16", expert="relu",
                                 dispatch_dtype="fp8_gemm"),
    "mixtral_fp8_experts": wl.scaled(W["mixtral_fp8_experts"], T=512, d=1024, F=1536),
    "decode_fp8_experts": wl.scaled(W["dsv3_decode"], d=1072, F=272, dispatch_dtype="fp8_gemm", precision="fp8_h"),
}


def stagewise(w, seed=0, inp=None):
    inp = wl.make_inputs(w, seed, device="cuda") if inp is None else inp
    cfg = abi.config_for(w)
    cap = capacity_of(cfg)
    st = wl.make_stage_inputs(w, seed, device="cuda", rows=abi.moe_rows_capacity(cfg))
    b = StageBuffers(w, cfg)
    b.route(inp)
    torch.cuda.synchronize()
    r = check_route(w, inp, b)
    d = check_dispatch(w, inp, b, cap, st)
    assert b.dispatch_status() == 0
    dd = check_dedup(w, inp, b, st, d) if w.dedup else None
    f8 = check_fp8(w, inp, b, st, d) if w.dispatch_dtype in ("fp8", "fp8_gemm") else None
    ffn_err = None
    if w.expert != "identity":
        ffn_err = check_ffn(w, inp, b, st)
        assert b.ffn_status() == 0
    comb_err = check_combine(w, b, st)
    assert abi.moe_read_status(b.status.data_ptr()) == 0
    c = chain(w, inp, cfg)
    chained = check_chained_dispatch(w, inp, c, r, cap)
    return dict(inp=inp, cfg=cfg, bufs=b, chain=c, route=r, dispatch=d, dedup=dd, ffn_err=ffn_err,
                combine_err=comb_err, chained=chained)


def layer_keep(w, ref, capacity):
    """Tokens compared end to end: no near tie in the router, and under the gate
    drop policy no gate at a keep cutoff."""
    keep = ~route_tie_flags(w, ref["H"])
    if w.drop_policy == "gate":
        keep &= ~gate_boundary_ties(w, ref["idx"][:, :w.k], ref["G"][:, :w.k], capacity)
    return keep


@pytest.mark.parametrize("name", list(REDUCED))
def test_stagewise_parity(name):
    w = REDUCED[name]
    res = stagewise(w)
    print(f"\n{name}: near-ties={res['route']['near_ties']} flipped={res['route']['flipped']} "
          f"gate_err={res['route']['gate_err']:.2e} ffn_err/rms={res['ffn_err']} "
          f"combine_err/rms={res['combine_err']:.2e} dropped={res['dispatch']['n_dropped']} "
          f"chained dispatch: {res['chained']}")


@pytest.mark.parametrize("name", list(REDUCED))
def test_layer_forward_matches_oracle(name):
    w = REDUCED[name]
    inp = wl.make_inputs(w, 1, device="cuda")
    cfg = abi.config_for(w)
    y, ws, view, flags = run_layer(cfg, inp, w)
    assert flags == 0
    ref = run_oracle(w, inp)
    keep = layer_keep(w, ref, capacity_of(cfg))
    extra = fp8_h_layer_budget(w, inp, ref)[keep] if w.precision == "fp8_h" else None
    err = check_layer_close(name, cpu(y)[torch.from_numpy(keep)], ref["y"][keep], w.act, f"{name} layer y",
                            extra=extra)
    print(f"\n{name}: layer max|err|/rms(y) = {err:.4f} (near-tie tokens excluded: {int((~keep).sum())})")
    if w.expert == "identity" and w.dispatch_dtype == "act":
        assert torch.equal(y, inp["x"]), "identity experts must return x exactly"


@pytest.mark.parametrize("name", ["grouped_dedup", "grouped_dedup_swiglu", "grouped_dedup_fp8",
                                  "grouped_dedup_fp8_swiglu", "grouped_dedup_fp8_gemm"])
def test_dedup_forward_equals_the_direct_forward_bitwise(name):
    """The deduplicated dispatch changes where rows travel, not their values: the layer
    output is the same bits, and the send map in the workspace is the oracle's."""
    w = REDUCED[name]
    inp = wl.make_inputs(w, 17, device="cuda")
    y_dd, ws, view, flags = run_layer(abi.config_for(w), inp, w)
    y_direct, _, _, _ = run_layer(abi.config_for(wl.scaled(w, dedup=False)), inp, w)
    assert flags == 0 and torch.equal(y_dd, y_direct)
    idx = cpu(WorkspaceMap(w, abi.config_for(w), ws, view).topk_idx).numpy()
    pos = ws[view.pos - ws.data_ptr():view.pos - ws.data_ptr() + 4 * w.T * w.slots].view(torch.int32).cpu().numpy()
    s = orc.dedup_send(idx, pos, w.E, w.D)
    base = ws.data_ptr()
    send_offsets = ws[view.send_offsets - base:view.send_offsets - base + 4 * (w.D + 1)].view(torch.int32).cpu()
    np.testing.assert_array_equal(send_offsets.numpy(), s["send_offsets"])
    # each token touches at most topk_groups ranks when the groups are the ranks
    assert int(s["sent"].sum(axis=1).max()) <= w.topk_groups
    print(f"\n{name}: rows sent {s['n_send']} for {int((pos >= 0).sum())} kept assignments "
          f"({s['n_send'] / w.T:.2f} ranks per token)")


def test_identity_experts_return_x_exactly_with_drops_zeroed():
    w = wl.Workload("ident_cap", T=1000, d=256, E=16, k=4, F=0, act="bf16", expert="identity",
                    capacity_factor="0.5", D=4)
    inp = wl.make_inputs(w, 2, device="cuda")
    cfg = abi.config_for(w)
    y, ws, view, flags = run_layer(cfg, inp, w)
    ref = run_oracle(w, inp)
    # with drops the layer returns x scaled by the kept gates' sum, once rounded
    check_close(y, ref["y"], "bf16", "identity with drops", tol=1e-5, with_half_ulp=True)
    assert ref["n_dropped"] > 0


def test_deterministic_bitwise():
    w = REDUCED["dsv3_full"]
    inp = wl.make_inputs(w, 3, device="cuda")
    cfg = abi.config_for(w)
    y1, ws1, _, _ = run_layer(cfg, inp, w)
    y2, ws2, _, _ = run_layer(cfg, inp, w)
    assert torch.equal(y1, y2)
    n = abi.moe_workspace_bytes(cfg)
    assert torch.equal(ws1[:n], ws2[:n]) or _ws_equal_used(cfg, ws1, ws2)


def _ws_equal_used(cfg, ws1, ws2):
    v1, v2 = abi.moe_workspace_get_view(cfg, ws1), abi.moe_workspace_get_view(cfg, ws2)
    base1, base2 = ws1.data_ptr(), ws2.data_ptr()
    A = cfg.T * (cfg.k + cfg.n_shared)
    for name, nbytes in [("topk_idx", 4 * A), ("topk_gate", 4 * A), ("pos", 4 * A), ("offsets", 4 * (cfg.E + 1))]:
        o1 = getattr(v1, name) - base1
        o2 = getattr(v2, name) - base2
        if not torch.equal(ws1[o1:o1 + nbytes], ws2[o2:o2 + nbytes]):
            return False
    return True


# Edge layers. Small layers with heavy-tailed outputs (few tokens, long rows, drops) can
# spend most of the 2e-2 * rms(y) budget on y's own bf16 rounding, and then the bf16
# rounding of h tips them over: those carry h as a hi/lo pair (precision "split_h"),
# which leaves y's rounding as the only error of size.
EDGE = [
    wl.Workload("T1_k1", T=1, d=64, E=4, k=1, F=64, act="bf16", expert="swiglu"),
    wl.Workload("k_eq_E", T=77, d=128, E=6, k=6, F=96, act="bf16", expert="swiglu", D=3),
    wl.Workload("E_not_pow2_ragged", T=333, d=136, E=12, k=3, F=200, act="bf16", expert="swiglu", D=4),
    wl.Workload("relu_bf16", T=300, d=192, E=5, k=2, F=320, act="bf16", expert="relu"),
    wl.Workload("swiglu_f32", T=200, d=96, E=7, k=3, F=72, act="f32", expert="swiglu"),
    wl.Workload("empty_experts", T=5, d=64, E=64, k=2, F=128, act="bf16", expert="swiglu", D=8),
    wl.Workload("zero_capacity", T=64, d=64, E=8, k=2, F=64, act="bf16", expert="swiglu", capacity_factor="0"),
    wl.Workload("cap_below_mean", T=600, d=128, E=8, k=2, F=128, act="bf16", expert="swiglu",
                capacity_factor="0.75", min_capacity=10),
    wl.Workload("cap_huge", T=64, d=64, E=8, k=2, F=64, act="bf16", expert="swiglu", capacity_factor="100",
                precision="split_h"),
    wl.Workload("k16_E256", T=96, d=256, E=256, k=16, F=128, act="bf16", expert="swiglu", D=8),
    wl.Workload("long_rows", T=130, d=8192, E=4, k=2, F=256, act="bf16", expert="swiglu", precision="split_h"),
    wl.Workload("split_h_relu", T=300, d=192, E=5, k=2, F=320, act="bf16", expert="relu", precision="split_h"),
    wl.Workload("split_h_ragged", T=333, d=136, E=12, k=3, F=192, act="bf16", expert="swiglu", D=4,
                precision="split_h", capacity_factor="0.9"),
    wl.Workload("gate_drops_ragged", T=333, d=136, E=12, k=3, F=192, act="bf16", expert="swiglu", D=4,
                capacity_factor="0.75", drop_policy="gate", zipf_s=1.2, precision="split_h"),
    wl.Workload("padded_token_order", T=300, d=128, E=8, k=2, F=128, act="bf16", expert="swiglu",
                capacity_factor="1", layout="padded", zipf_s=1.2, precision="split_h"),
    wl.Workload("padded_gate_f32", T=257, d=96, E=7, k=3, F=72, act="f32", expert="relu",
                capacity_factor="1.25", drop_policy="gate", layout="padded", zipf_s=1.2),
    wl.Workload("padded_zero_capacity", T=64, d=64, E=8, k=2, F=64, act="bf16", expert="swiglu",
                capacity_factor="0", layout="padded"),
    wl.Workload("padded_cap_huge", T=64, d=64, E=8, k=2, F=64, act="bf16", expert="swiglu",
                capacity_factor="100", layout="padded", drop_policy="gate", precision="split_h"),
    wl.Workload("padded_identity_gate", T=500, d=256, E=16, k=4, F=0, act="bf16", expert="identity",
                capacity_factor="0.5", D=4, layout="padded", drop_policy="gate"),
    # the FP8 up projection: one token, every expert per token, zero and huge capacity in
    # the padded layout, heavy drops with h as a hi/lo pair, rows longer than a stage ring
    wl.Workload("fp8_gemm_T1_k1", T=1, d=64, E=4, k=1, F=64, act="bf16", expert="swiglu",
                dispatch_dtype="fp8_gemm"),
    wl.Workload("fp8_gemm_k_eq_E", T=77, d=128, E=6, k=6, F=96, act="bf16", expert="swiglu", D=3,
                dispatch_dtype="fp8_gemm"),
    wl.Workload("fp8_gemm_padded_zero_capacity", T=64, d=64, E=8, k=2, F=64, act="bf16", expert="swiglu",
                capacity_factor="0", layout="padded", dispatch_dtype="fp8_gemm"),
    wl.Workload("fp8_gemm_padded_cap_huge", T=64, d=64, E=8, k=2, F=64, act="bf16", expert="relu",
                capacity_factor="100", layout="padded", drop_policy="gate", dispatch_dtype="fp8_gemm"),
    wl.Workload("fp8_gemm_split_h_drops", T=333, d=144, E=12, k=3, F=192, act="bf16", expert="swiglu", D=4,
                precision="split_h", capacity_factor="0.6", zipf_s=1.2, dispatch_dtype="fp8_gemm"),
    wl.Workload("fp8_gemm_long_rows", T=130, d=8192, E=4, k=2, F=256, act="bf16", expert="swiglu",
                dispatch_dtype="fp8_gemm", precision="split_h"),
]


@pytest.mark.parametrize("name", ["mixtral_bf16", "zipf_cf125", "dsv3_full"])
def test_split_h_mode_is_limited_by_the_output_rounding(name):
    """With h as a hi/lo pair and fp32 expert outputs, y is the exact result up to
    its own bf16 rounding plus a small fp32 residue."""
    w = wl.scaled(REDUCED[name], precision="split_h")
    inp = wl.make_inputs(w, 8, device="cuda")
    cfg = abi.config_for(w)
    y, ws, view, flags = run_layer(cfg, inp, w)
    assert flags == 0
    ref = run_oracle(w, inp)
    s, o = orc.near_tie_flags(ref["H"], w.k)
    keep = ~(s | o)
    err = check_close(cpu(y)[torch.from_numpy(keep)], ref["y"][keep], "bf16", f"{name} split-h y", tol=2e-3,
                      with_half_ulp=True)
    print(f"\n{name} split_h: raw max|err|/rms(y) = {err:.4f}")


@pytest.mark.parametrize("name", ["mixtral_bf16", "dsv3_full", "mixtral_fp8_gemm"])
def test_bf16_mode_within_its_rounding_budget(name):
    """All-bf16 mode: the expert outputs are rounded to bf16 too, so the bound adds
    their half-ulp, weighted by the gates, to the f32-output bound. (Dropless layers
    only: with heavy drops rms(y) shrinks and the h rounding alone exceeds 2e-2*rms,
    which is why the capacity workload runs with h split into a hi/lo pair.)"""
    w = wl.scaled(REDUCED[name], precision="bf16")
    inp = wl.make_inputs(w, 9, device="cuda")
    cfg = abi.config_for(w)
    y, ws, view, flags = run_layer(cfg, inp, w)
    assert flags == 0
    ref = run_oracle(w, inp)
    s, o = orc.near_tie_flags(ref["H"], w.k)
    keep = ~(s | o)
    out_half_ulp = half_ulp(ref["out"], "bf16")
    extra = orc.combine(ref["G"], ref["pos"], out_half_ulp, w.T, w.slots)
    got, exact = f64(y)[keep], ref["y"][keep]
    err = np.abs(got - exact)
    bound = 2e-2 * rms(exact) + half_ulp(exact, "bf16") + extra[keep]
    assert np.all(err <= bound), f"{name}: worst excess {(err - bound).max():.3e}"


@pytest.mark.parametrize("w", EDGE, ids=[w.name for w in EDGE])
def test_edge_cases(w):
    res = stagewise(w, seed=4)
    inp, cfg = res["inp"], res["cfg"]
    y, ws, view, flags = run_layer(cfg, inp, w)
    assert flags == 0
    assert torch.equal(y, res["chain"].y), "layer and chained stage calls must agree bit for bit"
    ref = run_oracle(w, inp)
    keep = layer_keep(w, ref, capacity_of(cfg))
    check_layer_close(w.name, cpu(y)[torch.from_numpy(keep)], ref["y"][keep], w.act, f"{w.name} layer y")
    if w.capacity_factor == "0":
        assert torch.count_nonzero(y) == 0


@pytest.mark.parametrize("E", [8, 64])
def test_near_tie_count_with_duplicated_router_columns(E):
    """Two identical columns of W_g give two exactly equal logits on every token, so
    each token that ranks them k-th and (k+1)-th is a near tie the forward must count
    (within the band of check_near_tie_count); the fused small-E router (E = 8) and
    the split-K router (E = 64) each count their own."""
    w = wl.Workload(f"dup_cols_E{E}", T=3000, d=256, E=E, k=2, F=0, act="bf16", expert="identity")
    inp = wl.make_inputs(w, 21, device="cuda")
    inp["Wg"][:, 5] = inp["Wg"][:, 3]
    cfg = abi.config_for(w)
    y, ws, view, flags = run_layer(cfg, inp, w)
    assert flags == 0
    H = orc.router_logits(f64(inp["x"]), f64(inp["Wg"]), None)
    s = -np.sort(-H, axis=1)
    planted = int(((s[:, w.k - 1] == s[:, w.k]) & (s[:, w.k] != 0)).sum())
    n = check_near_tie_count(w, ws, view, H)
    assert planted > 0 and n >= planted, (n, planted)
    print(f"\nE={E}: {n} near-tie tokens counted, {planted} of them planted exact ties")


def test_all_tokens_to_one_expert_with_capacity():
    w = wl.Workload("hot", T=512, d=128, E=8, k=1, F=128, act="bf16", expert="swiglu", capacity_factor="1")
    inp = wl.make_inputs(w, 5, device="cuda")
    inp["bias"] = torch.tensor([0, 0, 0, 1000.0, 0, 0, 0, 0], device="cuda")
    res = stagewise(w, inp=inp)
    c = res["chain"]
    assert res["chained"] == "exact"
    assert int(c.counts_routed[3]) == 512 and int(c.counts_kept[3]) == 64 and int(c.n_dropped[0]) == 448


def test_host_buffer_path_matches_device_path():
    w = REDUCED["mixtral_bf16"]
    inp = wl.make_inputs(w, 6, device="cuda")
    cfg = abi.config_for(w)
    y_dev, _, _, _ = run_layer(cfg, inp, w)
    ws = abi.workspace(cfg, host=True)
    x_host = inp["x"].cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    abi.moe_layer_forward_host(cfg, x_host, inp["Wg"], None, inp["W13"], inp["W2"], y_host, ws)
    assert torch.equal(y_host, y_dev.cpu())


def test_traced_forward_matches_and_times():
    w = REDUCED["mixtral_bf16"]
    inp = wl.make_inputs(w, 7, device="cuda")
    cfg = abi.config_for(w)
    y_dev, _, _, _ = run_layer(cfg, inp, w)
    ws = abi.workspace(cfg)
    y = torch.empty_like(y_dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    abi.moe_layer_forward_traced(cfg, inp["x"], inp["Wg"], None, inp["W13"], inp["W2"], y, ws, ev)
    torch.cuda.synchronize()
    assert torch.equal(y, y_dev)
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(t >= 0 for t in times) and sum(times) > 0


# ------------------------------------------------------------------ full sizes, sampled
def _sampled_y(w, inp, ref_route, disp, tokens):
    """Oracle y for a few tokens from the full-batch routing and dispatch (drops included);
    with the FP8 dispatch routed experts see the dequantized rows. Also returns the FP8
    hidden-activation budget of those tokens (zeros unless the precision is fp8_h)."""
    x = f64(inp["x"][torch.as_tensor(tokens, device="cuda")])
    xq = orc.quantize_fp8_blocks(x)["deq"] if w.dispatch_dtype == "fp8" else x
    fp8_gemm = w.dispatch_dtype == "fp8_gemm"
    if fp8_gemm:  # every row, shared ones too, is the row-quantized token
        x = xq = orc.quantize_fp8_rows(x)["deq"]
    idx, G, pos = ref_route["idx"], ref_route["G"], disp["pos"].reshape(w.T, w.slots)
    # the FP8 hidden activation's budget reuses the quantized weights (kept for that layer only:
    # the float64 weights of every expert of the larger layers would not fit the host)
    fn = expert_fn(w.expert, inp["W13"], inp["W2"], w.F, fp8_up=fp8_gemm, fp8_h=w.precision == "fp8_h",
                   cache=inp.setdefault("_expert_cache", {}) if w.precision == "fp8_h" else None)
    need = {}
    for r, t in enumerate(tokens):
        for j in range(w.slots):
            if pos[t, j] >= 0:
                need.setdefault(int(idx[t, j]), []).append((r, j))
    y = np.zeros((len(tokens), w.d))
    budget = np.zeros_like(y)
    for e, uses in need.items():
        rows = np.array([r for r, _ in uses])
        xin = (xq if e < w.E else x)[rows]
        outs = fn(e, xin)
        b = fp8_h_budget(w, inp, e, xin) if w.precision == "fp8_h" else np.zeros_like(outs)
        for (r, j), o, bo in zip(uses, outs, b):
            y[r] += G[tokens[r], j] * o
            budget[r] += G[tokens[r], j] * bo
    return y, budget


FULL = {n: W[n] for n in ["mixtral_bf16", "dsv3_route_only", "zipf_cf125", "dsv3_full", "dsv3_decode"]}
FULL["zipf_gate_padded"] = wl.scaled(W["zipf_cf125"], drop_policy="gate", layout="padded")
FULL["dsv3_grouped_dedup"] = W["dsv3_grouped_dedup"]
FULL["mixtral_fp8_dispatch"] = W["mixtral_fp8_dispatch"]
FULL["mixtral_fp8_gemm"] = W["mixtral_fp8_gemm"]
FULL["dsv3_decode_fp8_gemm"] = W["dsv3_decode_fp8_gemm"]
FULL["mixtral_fp8_experts"] = W["mixtral_fp8_experts"]
FULL["dsv3_grouped_dedup_fp8"] = W["dsv3_grouped_dedup_fp8"]
FULL["dsv3_full_fp8_gemm_dedup"] = W["dsv3_full_fp8_gemm_dedup"]


# Tokens whose y is compared element by element at full size: 256 on the DeepSeek-V3-shaped
# layer, 64 on the others, fewer on the FP8-GEMM layers (below).
SAMPLED_TOKENS = 256
SAMPLED_TOKENS_OTHERS = 64


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(name):
    w = FULL[name]
    inp = wl.make_inputs(w, 0, device="cuda")
    cfg = abi.config_for(w)
    cap = capacity_of(cfg)
    y, ws, view, flags = run_layer(cfg, inp, w)
    assert flags == 0
    m = WorkspaceMap(w, cfg, ws, view)
    # router: full oracle logits in float64, and the forward's own near-tie count
    r = check_route(w, inp, m)
    n_ties = check_near_tie_count(w, ws, view, r["H"])
    # the GPU dispatch of the oracle's routing: bit-exact at full size, always
    check_dispatch_of_oracle_routing(w, inp, cfg, r, cap)
    # dispatch of the GPU's routing: bit-exact against the oracle's where the routings agree
    how = check_chained_dispatch(w, inp, m, r, cap)
    d = oracle_dispatch(w, r["idx_full"], r["G_full"], cap)
    if w.dedup and how == "exact":
        s = orc.dedup_send(r["idx_full"], d["pos"], w.E, w.D)
        np.testing.assert_array_equal(cpu(m.send_offsets).numpy(), s["send_offsets"])
        np.testing.assert_array_equal(cpu(m.send_pos).numpy(), s["send_pos"])
        np.testing.assert_array_equal(cpu(m.send_src).numpy()[:s["n_send"]], s["send_src"])
        src = torch.from_numpy(s["send_src"] // w.D).cuda()
        if w.dispatch_dtype == "fp8":  # codes and block scales of 64 sampled send rows
            rows = np.random.default_rng(3).choice(s["n_send"], size=min(64, s["n_send"]), replace=False)
            q = orc.quantize_fp8_blocks(f64(inp["x"][src[torch.from_numpy(rows).cuda()]]))
            np.testing.assert_array_equal(cpu(m.xsend).numpy()[rows], q["codes"])
            np.testing.assert_array_equal(cpu(m.xsend_scale).numpy().astype(np.float64)[rows], q["scales"])
        elif w.dispatch_dtype == "fp8_gemm":  # codes and row scales of 64 sampled send rows
            rows = np.random.default_rng(3).choice(s["n_send"], size=min(64, s["n_send"]), replace=False)
            q = orc.quantize_fp8_rows(f64(inp["x"][src[torch.from_numpy(rows).cuda()]]))
            np.testing.assert_array_equal(cpu(m.xsend).numpy()[rows], q["codes"])
            np.testing.assert_array_equal(cpu(m.xsend_scale).numpy().astype(np.float64).reshape(-1)[rows],
                                          q["scales"])
        else:
            assert torch.equal(m.xsend[:s["n_send"]], inp["x"][src])
        print(f"\n{name}: {s['n_send']} send rows, {s['n_send'] / w.T:.3f} ranks per token")
    fp8 = w.dispatch_dtype == "fp8"
    if fp8 and how == "exact" and not w.dedup:
        # codes and scales of 64 sampled routed rows against the oracle's quantization
        rows = np.nonzero(d["row_src"] >= 0)[0]
        rows = np.random.default_rng(1).choice(rows, size=min(64, rows.size), replace=False)
        tok = d["row_src"][rows] // w.slots
        q = orc.quantize_fp8_blocks(f64(inp["x"][torch.from_numpy(tok).cuda()]))
        np.testing.assert_array_equal(cpu(m.xq).numpy()[rows], q["codes"])
        np.testing.assert_array_equal(cpu(m.xscale).numpy().astype(np.float64)[rows], q["scales"])
    if w.dispatch_dtype == "fp8_gemm" and how == "exact":
        # the FP8 GEMM's input rows (with dedup: as the fan-out wrote them) on 64 sampled rows
        rows = np.nonzero(d["row_src"] >= 0)[0]
        rows = np.random.default_rng(1).choice(rows, size=min(64, rows.size), replace=False)
        compare_fp8_rows(w, m.xq, m.xscale, d["row_src"], inp["x"], rows=rows)
    if w.expert == "identity" and w.dispatch_dtype == "act":
        assert torch.equal(y, inp["x"])
        return
    # expert outputs of a few whole experts (largest, smallest non-empty, two more); with
    # an exact dispatch their input rows are x at the oracle's row sources (FP8 dispatch:
    # the dequantized rows)
    worst_ffn = None
    if how == "exact":
        counts = d["counts_kept"]
        nz = np.nonzero(counts)[0]
        pick = sorted({int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])]), int(nz[len(nz) // 2]),
                       int(nz[0])})
        if w.precision == "fp8_h":  # the code-flip budget costs a second pass per expert: two experts
            pick = sorted({int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])})
        fp8_gemm = w.dispatch_dtype == "fp8_gemm"
        fn = expert_fn(w.expert, inp["W13"], inp["W2"], w.F, fp8_up=fp8_gemm, fp8_h=w.precision == "fp8_h",
                       cache=inp.setdefault("_expert_cache", {}) if w.precision == "fp8_h" else None)
        worst_ffn = 0.0
        for e in pick:
            lo = int(d["offsets"][e])
            hi = lo + int(counts[e])
            src = torch.from_numpy(d["row_src"][lo:hi] // w.slots).cuda()
            xin = f64(inp["x"][src])
            if fp8 and e < w.E:
                xin = orc.quantize_fp8_blocks(xin)["deq"]
            if fp8_gemm:
                xin = orc.quantize_fp8_rows(xin)["deq"]
            extra = fp8_h_budget(w, inp, e, xin) if w.precision == "fp8_h" else None
            worst_ffn = max(worst_ffn, check_close(m.out[lo:hi], fn(e, xin), m.out_act, f"expert {e}", tol=2e-2,
                                                   extra=extra))
    # end to end on sampled tokens from the oracle's own routing and dispatch: no near
    # tie, no gate at a keep cutoff, and (with a capacity) no expert shared with a
    # token whose routing flipped
    ok = ~r["tie"]
    if w.drop_policy == "gate":
        ok &= ~gate_boundary_ties(w, r["idx"], r["G"], cap)
    idx_g = cpu(m.topk_idx).numpy()[:, :w.k]
    flipped = (idx_g != r["idx"]).any(axis=1)
    if flipped.any() and cap is not None:
        touched = set(r["idx"][flipped].ravel().tolist()) | set(idx_g[flipped].ravel().tolist())
        ok &= ~np.isin(r["idx"], sorted(touched)).any(axis=1)
    ok &= ~flipped
    rng = np.random.default_rng(0)
    cand = np.nonzero(ok)[0]
    n_tok = SAMPLED_TOKENS if name == "dsv3_full" else SAMPLED_TOKENS_OTHERS
    if w.dispatch_dtype == "fp8_gemm" and w.expert != "identity":
        # the oracle quantizes every expert a sampled token uses (2F x d weights each, in
        # float64): 8 tokens, 4 on the DeepSeek-V3-shaped layers (8 or 9 experts per token)
        n_tok = 4 if (w.T <= 128 or w.E >= 256) else 8
    tokens = sorted(rng.choice(cand, size=min(n_tok, cand.size), replace=False).tolist())
    y_s, budget = _sampled_y(w, inp, dict(idx=r["idx_full"], G=r["G_full"]), d, tokens)
    err = check_layer_close(name, y[torch.as_tensor(tokens, device="cuda")], y_s, w.act, f"{name} sampled y",
                            extra=budget, whole=False)
    print(f"\n{name}: near-ties={r['near_ties']} (GPU count of k-th/(k+1)-th ties: {n_ties}) flipped={r['flipped']} "
          f"dispatch={how} ffn_err/rms={worst_ffn} sampled y err/rms={err:.4f} over {len(tokens)} tokens "
          f"dropped={d['n_dropped']}")


@pytest.mark.parametrize("name", ["mixtral_bf16", "zipf_cf125", "tiny_f32"])
def test_layer_forward_replays_in_a_cuda_graph(name):
    """The whole forward enqueues without host syncs, so it captures into a CUDA
    graph; replays on new inputs equal eager calls bit for bit."""
    w = REDUCED[name]
    cfg = abi.config_for(w)
    inp = wl.make_inputs(w, 14, device="cuda")
    ws = abi.workspace(cfg)
    y = torch.empty(w.T, w.d, dtype=w.torch_act, device="cuda")
    fwd = lambda: abi.moe_layer_forward(cfg, inp["x"], inp["Wg"], inp.get("bias"), inp.get("W13"), inp.get("W2"),
                                        y, ws)
    fwd()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fwd()
    for seed in (15, 16):
        new = wl.make_inputs(w, seed, device="cuda")
        inp["x"].copy_(new["x"])
        g.replay()
        torch.cuda.synchronize()
        y_graph = y.clone()
        fwd()
        torch.cuda.synchronize()
        assert torch.equal(y_graph, y)


def test_forward_from_two_host_threads_shares_the_context_setup():
    """Kernel attributes, cluster occupancy and the static dispatch scratch address are set
    up once per CUDA context and then looked up: two host threads calling the layer (and the
    static dispatch) on the same device, each on its own stream, must find that setup and
    give the same bits as one thread does."""
    import threading
    w = REDUCED["dsv3_full"]
    inp = wl.make_inputs(w, 19, device="cuda")
    cfg = abi.config_for(w)
    y_ref, _, _, _ = run_layer(cfg, inp, w)
    torch.cuda.synchronize()
    results, errors = {}, []
    static_lock = threading.Lock()  # static-dispatch calls share one scratch array: never overlap them

    def worker(i):
        try:
            torch.cuda.set_device(0)
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                ws = abi.workspace(cfg)
                y = torch.empty_like(y_ref)
                for _ in range(3):
                    abi.moe_layer_forward(cfg, inp["x"], inp["Wg"], None, inp["W13"], inp["W2"], y, ws,
                                          stream=stream)
                b = StageBuffers(w, cfg)
                b.route(inp)
                with static_lock:
                    abi.moe_dispatch_static(cfg, inp["x"], b.topk_idx, b.dmap(), b.xperm, stream=stream,
                                            topk_gate=b.topk_gate)
                    stream.synchronize()
            stream.synchronize()
            results[i] = (y, b)
        except Exception as exc:  # noqa: BLE001 - reported below
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert abi.lib().moe_last_cuda_error() in (b"", None)
    for i in range(2):
        y, b = results[i]
        assert torch.equal(y, y_ref)
    assert torch.equal(results[0][1].offsets, results[1][1].offsets)
    assert torch.equal(results[0][1].pos, results[1][1].pos)


def test_async_host_forward_on_two_streams_matches_the_device_forward():
    w = REDUCED["mixtral_bf16"]
    inp = wl.make_inputs(w, 18, device="cuda")
    cfg = abi.config_for(w)
    y_dev, _, _, _ = run_layer(cfg, inp, w)
    x_host = inp["x"].cpu().pin_memory()
    ws = [abi.workspace(cfg, host=True) for _ in range(2)]
    ys = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    for i in range(4):
        abi.moe_layer_forward_host_async(cfg, x_host, inp["Wg"], None, inp["W13"], inp["W2"], ys[i % 2], ws[i % 2],
                                         streams[i % 2])
    for st in streams:
        st.synchronize()
    assert torch.equal(ys[0], y_dev.cpu()) and torch.equal(ys[1], y_dev.cpu())
