"""Pins for the CPU oracle: each test checks it against something other than itself.

The pins come from the gating equations (closed forms, special cases that reduce
to a library routine), brute force on tiny inputs, invariants the method fixes
(gates sum to one, counts add up, identity experts return x) and exact small
constructions. They are chosen so that a dropped term, a flipped sign or index, a
transposed operand or a wrong ordering rule fails at least one of them.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as Fn

from oracle import moe_oracle as orc
from routing_dispatch_combine_moe_b300 import workloads as wl
from tests._harness import expert_fn, f64, run_oracle


def rng(seed=0):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------- KeepTopK
@pytest.mark.parametrize("E,k", [(2, 1), (3, 2), (5, 2), (6, 3), (8, 2), (9, 4), (10, 5), (10, 10)])
def test_topk_matches_brute_force_subsets(E, k):
    """The kept set is the only k-subset whose minimum beats every excluded value."""
    r = rng(E * 31 + k)
    H = r.normal(size=(50, E))
    idx = orc.keep_topk(H, k)
    for t in range(H.shape[0]):
        winners = [
            S for S in itertools.combinations(range(E), k)
            if all(min(H[t, list(S)]) > H[t, o] for o in range(E) if o not in S)
        ]
        assert len(winners) == 1
        assert set(idx[t].tolist()) == set(winners[0])
        vals = H[t, idx[t]]
        assert np.all(np.diff(vals) < 0), "slots must be in descending logit order"


def test_topk_ties_prefer_lower_expert_id():
    H = np.array([[1.0, 3.0, 3.0, 2.0],
                  [0.5, 0.5, 0.5, 0.5],
                  [-1.0, 2.0, -1.0, 2.0]])
    assert orc.keep_topk(H, 2).tolist() == [[1, 2], [0, 1], [1, 3]]
    assert orc.keep_topk(H, 3).tolist() == [[1, 2, 3], [0, 1, 2], [1, 3, 0]]
    assert orc.keep_topk(H, 1).tolist() == [[1], [0], [1]]


def test_topk_k_equals_E_is_full_descending_sort():
    H = rng(1).normal(size=(20, 7))
    idx = orc.keep_topk(H, 7)
    np.testing.assert_array_equal(idx, np.argsort(-H, axis=1, kind="stable"))


# ----------------------------------------------------------------------- gates
def test_gates_with_k_equal_E_are_the_full_softmax():
    H = rng(2).normal(size=(30, 9)) * 3
    idx = orc.keep_topk(H, 9)
    G = orc.kept_softmax(H, idx)
    full = scipy.special.softmax(H, axis=1)
    np.testing.assert_allclose(G, np.take_along_axis(full, idx, axis=1), rtol=1e-14, atol=0)


def test_gates_closed_form_two_kept_of_three():
    """Kept logits a > b, third logit excluded: G = (1/(1+e^(b-a)), 1/(1+e^(a-b)))."""
    a, b, c = 1.7, -0.4, 1.2  # c sits between: keep top-2 = {a, c}
    H = np.array([[a, b, c]])
    idx = orc.keep_topk(H, 2)
    assert idx.tolist() == [[0, 2]]
    G = orc.kept_softmax(H, idx)[0]
    assert G[0] == pytest.approx(1 / (1 + math.exp(c - a)), rel=1e-15)
    assert G[1] == pytest.approx(1 / (1 + math.exp(a - c)), rel=1e-15)


def test_gates_k1_are_one_and_sum_to_one():
    H = rng(3).normal(size=(40, 16)) * 5
    for k in (1, 2, 5, 16):
        G = orc.kept_softmax(H, orc.keep_topk(H, k))
        np.testing.assert_allclose(G.sum(axis=1), 1.0, rtol=0, atol=4e-16)
        assert np.all(np.diff(G, axis=1) <= 0), "gates follow the descending logits"
    assert np.all(orc.kept_softmax(H, orc.keep_topk(H, 1)) == 1.0)


def test_gates_are_shift_invariant_and_large_logits_finite():
    H = rng(4).normal(size=(10, 8))
    idx = orc.keep_topk(H, 3)
    np.testing.assert_allclose(orc.kept_softmax(H + 700.0, idx), orc.kept_softmax(H, idx), rtol=1e-12)


def test_router_logits_bias_enters_selection_and_gates():
    """A large bias on expert 2 puts it first for every token; its gate follows the biased logit."""
    x = rng(5).normal(size=(6, 4))
    Wg = rng(6).normal(size=(4, 5))
    bias = np.array([0.0, 0.0, 50.0, 0.0, 0.0])
    H = orc.router_logits(x, Wg, bias)
    np.testing.assert_allclose(H, x @ Wg + bias, rtol=1e-15)
    idx = orc.keep_topk(H, 2)
    assert np.all(idx[:, 0] == 2)
    G = orc.kept_softmax(H, idx)
    assert np.all(G[:, 0] > 0.999)


def test_router_logits_match_torch_matmul():
    x = rng(7).normal(size=(33, 70))
    Wg = rng(8).normal(size=(70, 12))
    ref = torch.from_numpy(x) @ torch.from_numpy(Wg)
    np.testing.assert_allclose(orc.router_logits(x, Wg), ref.numpy(), rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------- near ties
def test_near_tie_flags():
    H = np.array([[3.0, 2.0, 2.0 * (1 - 3e-7), 0.0],   # k=2: 2nd vs 3rd within 1e-6 -> set tie
                  [3.0, 3.0 * (1 - 1e-7), 1.0, 0.0],   # 1st vs 2nd within 1e-6 -> order tie
                  [3.0, 2.0, 1.0, 0.0]])
    s, o = orc.near_tie_flags(H, 2)
    assert s.tolist() == [True, False, False]
    assert o.tolist() == [False, True, False]
    s, o = orc.near_tie_flags(H, 4)
    assert not s.any()


# ----------------------------------------------------------------------- capacity
def test_capacity_round_up_and_floor():
    assert orc.expert_capacity(8192, 2, 64, "1.25") == 320
    assert orc.expert_capacity(10, 1, 3, 1) == 4  # 10/3 rounds up
    assert orc.expert_capacity(10, 1, 3, "0.9") == 3  # 9/3 exactly
    assert orc.expert_capacity(10, 1, 3, "0.91") == 4
    assert orc.expert_capacity(16, 2, 8, "1.0") == 4
    assert orc.expert_capacity(16, 2, 8, "1.0", min_capacity=6) == 6
    assert orc.expert_capacity(16, 2, 8, 0) == 0
    assert orc.expert_capacity(16, 2, 8, None) is None


# ----------------------------------------------------------------------- dispatch
def _brute_dispatch(idx, E, C):
    """Expected rows from a plain sort of (expert, token, slot) triples."""
    T, k = idx.shape
    triples = sorted((int(idx[t, j]), t, j) for t in range(T) for j in range(k))
    rows, drops, seen = [], [], {}
    for e, t, j in triples:
        n = seen.get(e, 0)
        seen[e] = n + 1
        (rows if C is None or n < C else drops).append(t * k + j)
    return rows, drops


@pytest.mark.parametrize("C", [None, 0, 1, 3, 7, 1000])
def test_dispatch_matches_sorted_triples(C):
    r = rng(11)
    T, E, k = 37, 6, 3
    idx = np.stack([r.permutation(E)[:k] for _ in range(T)])
    disp = orc.dispatch(idx, E, C, D=2)
    rows, drops = _brute_dispatch(idx, E, C)
    assert disp["row_src"].tolist() == rows
    assert disp["drop_list"].tolist() == drops
    assert disp["n_dropped"] == len(drops)
    routed = np.bincount(idx.ravel(), minlength=E)
    np.testing.assert_array_equal(disp["counts_routed"], routed)
    kept = routed if C is None else np.minimum(routed, C)
    np.testing.assert_array_equal(disp["counts_kept"], kept)
    assert disp["counts_routed"].sum() == T * k
    assert disp["counts_kept"].sum() == T * k - disp["n_dropped"]
    np.testing.assert_array_equal(disp["offsets"], np.concatenate([[0], np.cumsum(kept)]))
    # pos and row_src are inverse on kept rows; dropped assignments are -1
    pos = disp["pos"]
    assert np.all(pos[disp["row_src"]] == np.arange(len(rows)))
    assert np.all(pos[disp["drop_list"]] == -1)
    assert (pos >= 0).sum() == len(rows)
    # D = 2 virtual ranks own experts [0,3) and [3,6)
    off = disp["offsets"]
    assert disp["rank_offsets"].tolist() == [0, off[3], off[6]]


def test_dispatch_all_tokens_to_one_expert():
    T, E, k = 20, 4, 1
    idx = np.zeros((T, k), np.int64)
    d = orc.dispatch(idx, E, capacity=5)
    assert d["counts_routed"].tolist() == [20, 0, 0, 0]
    assert d["counts_kept"].tolist() == [5, 0, 0, 0]
    assert d["row_src"].tolist() == [0, 1, 2, 3, 4]
    assert d["drop_list"].tolist() == list(range(5, 20))


# ----------------------------------------------------------------------- experts
def test_swiglu_closed_form_scalar():
    """d = F = 1: y = silu(x wg) (x wu) wd with silu(z) = z / (1 + e^-z)."""
    x, wg, wu, wd = 1.5, 2.0, -3.0, 0.5
    got = orc.expert_swiglu(np.array([[x]]), np.array([[wg]]), np.array([[wu]]), np.array([[wd]]))
    z = x * wg
    assert got[0, 0] == pytest.approx(z / (1 + math.exp(-z)) * (x * wu) * wd, rel=1e-15)
    # gate and up are not interchangeable
    swapped = orc.expert_swiglu(np.array([[x]]), np.array([[wu]]), np.array([[wg]]), np.array([[wd]]))
    assert abs(swapped[0, 0] - got[0, 0]) > 0.1


@pytest.mark.parametrize("kind", ["relu", "swiglu"])
def test_single_expert_k1_layer_is_the_ffn(kind):
    """E = 1, k = 1: the gate is 1 and the layer reduces to the FFN (torch as witness)."""
    w = wl.Workload("t", T=19, d=24, E=1, k=1, F=40, act="f32", expert=kind)
    inp = wl.make_inputs(w, seed=3)
    res = run_oracle(w, inp)
    x = inp["x"].double()
    W13, W2 = inp["W13"][0].double(), inp["W2"][0].double()
    if kind == "relu":
        ref = Fn.linear(Fn.relu(Fn.linear(x, W13)), W2)
    else:
        g, u = Fn.linear(x, W13[: w.F]), Fn.linear(x, W13[w.F:])
        ref = Fn.linear(Fn.silu(g) * u, W2)
    assert np.all(res["G"] == 1.0)
    np.testing.assert_allclose(res["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_combine_closed_form_with_a_drop():
    """Both tokens pick expert 0 first; C = 1 drops token 1's slot 0.

    Token 0 routes to (0, 1), token 1 to (0, 2). y_1 must be G[1,1] * Expert_2(x_1)
    alone: the dropped slot adds nothing and the surviving gate is not renormalised.
    """
    x = np.array([[1.0, 2.0], [3.0, -1.0]])
    Wg = np.array([[1.0, 0.0, 0.5], [0.5, 0.4, 0.0]])  # H0 = (2, .8, .5), H1 = (2.5, -.4, 1.5)
    scale = {0: 2.0, 1: -1.0, 2: 5.0}
    res = orc.moe_forward(x, Wg, 2, lambda e, X: scale[e] * X, capacity=1)
    H = x @ Wg
    assert res["idx"].tolist() == [[0, 1], [0, 2]]
    assert res["pos"].tolist() == [0, 1, -1, 2]
    assert res["drop_list"].tolist() == [2]
    g0 = (1 / (1 + math.exp(H[0, 1] - H[0, 0])), 1 / (1 + math.exp(H[0, 0] - H[0, 1])))
    g1 = (1 / (1 + math.exp(H[1, 2] - H[1, 0])), 1 / (1 + math.exp(H[1, 0] - H[1, 2])))
    np.testing.assert_allclose(res["y"][0], g0[0] * 2.0 * x[0] + g0[1] * -1.0 * x[0], rtol=1e-15)
    np.testing.assert_allclose(res["y"][1], g1[1] * 5.0 * x[1], rtol=1e-15)


def test_identity_experts_return_x_in_bf16():
    """Identity experts, dropless: y = x * sum(G) = x, exactly once rounded to bf16."""
    w = wl.Workload("t", T=300, d=64, E=16, k=4, F=0, act="bf16", expert="identity", D=4)
    inp = wl.make_inputs(w, seed=5)
    res = run_oracle(w, inp)
    np.testing.assert_array_equal(orc.round_to_bf16(res["y"]), f64(inp["x"]))


def test_zero_capacity_drops_everything_and_y_is_zero():
    w = wl.Workload("t", T=40, d=16, E=4, k=2, F=24, act="f32", expert="relu", capacity_factor="0")
    inp = wl.make_inputs(w, seed=6)
    res = run_oracle(w, inp)
    assert res["n_dropped"] == w.T * w.k
    assert np.all(res["y"] == 0.0)


def test_large_capacity_equals_dropless():
    w = wl.Workload("t", T=40, d=16, E=4, k=2, F=24, act="f32", expert="swiglu")
    inp = wl.make_inputs(w, seed=7)
    a = run_oracle(w, inp, capacity=None)
    b = run_oracle(w, inp, capacity=w.T * w.k)
    np.testing.assert_array_equal(a["y"], b["y"])
    assert b["n_dropped"] == 0


def test_expert_relabelling_leaves_y_unchanged():
    """Permuting expert ids (router columns and weights together) changes nothing in y."""
    w = wl.Workload("t", T=64, d=32, E=6, k=2, F=48, act="f32", expert="swiglu")
    inp = wl.make_inputs(w, seed=8)
    perm = torch.tensor([3, 0, 5, 1, 4, 2])
    inp2 = dict(inp, Wg=inp["Wg"][:, perm], W13=inp["W13"][perm], W2=inp["W2"][perm])
    a, b = run_oracle(w, inp), run_oracle(w, inp2)
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-13, atol=1e-13)


def test_dropless_tokens_are_independent():
    w = wl.Workload("t", T=50, d=32, E=8, k=3, F=40, act="f32", expert="relu")
    inp = wl.make_inputs(w, seed=9)
    full = run_oracle(w, inp)["y"]
    w1 = wl.Workload("t", T=1, d=32, E=8, k=3, F=40, act="f32", expert="relu")
    for t in (0, 17, 49):
        one = run_oracle(w1, dict(inp, x=inp["x"][t:t + 1]))["y"]
        np.testing.assert_allclose(one[0], full[t], rtol=1e-13, atol=1e-14)


def test_gates_scale_the_layer_linearly_in_w2():
    w = wl.Workload("t", T=30, d=16, E=4, k=2, F=24, act="f32", expert="relu")
    inp = wl.make_inputs(w, seed=10)
    a = run_oracle(w, inp)["y"]
    b = run_oracle(w, dict(inp, W2=inp["W2"] * 2))["y"]
    np.testing.assert_allclose(b, 2 * a, rtol=1e-13, atol=1e-14)


# ----------------------------------------------------------------------- bf16 rounding
def test_round_to_bf16_matches_torch_cast():
    r = rng(12)
    v = np.concatenate([r.normal(size=5000) * 10.0 ** r.integers(-6, 6, size=5000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 1e-40]])
    v32 = v.astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(orc.round_to_bf16(v32), ref)


# ----------------------------------------------------------------------- workload recipe
def test_zipf_workload_hot_expert_draws_forty_percent():
    w = wl.WORKLOADS["zipf_cf125"]
    x, Wg, bias = wl.make_router_inputs(w, 0)
    idx = orc.keep_topk(orc.router_logits(f64(x), f64(Wg), f64(bias)), w.k)
    share = np.bincount(idx.ravel(), minlength=w.E).max() / idx.size
    assert abs(share - 0.40) <= 0.01


# ----------------------------------------------------------------------- shared experts
def test_shared_expert_alone_is_the_ffn():
    """Routed experts' down projections zero: the layer reduces to the shared FFN (torch witness)."""
    w = wl.Workload("t", T=23, d=32, E=4, k=2, F=48, act="f32", expert="swiglu", n_shared=1)
    inp = wl.make_inputs(w, seed=21)
    inp["W2"][: w.E] = 0
    res = run_oracle(w, inp)
    x = inp["x"].double()
    W13, W2 = inp["W13"][w.E].double(), inp["W2"][w.E].double()
    ref = Fn.linear(Fn.silu(Fn.linear(x, W13[: w.F])) * Fn.linear(x, W13[w.F:]), W2)
    np.testing.assert_allclose(res["y"], ref.numpy(), rtol=1e-12, atol=1e-12)
    assert res["idx"].shape == (w.T, 3) and np.all(res["idx"][:, 2] == w.E) and np.all(res["G"][:, 2] == 1.0)


def test_shared_expert_adds_to_the_routed_layer():
    """y(shared) = y(routed only) + FFN_shared(x): with the shared expert's W2 zero they agree."""
    w1 = wl.Workload("t", T=40, d=32, E=6, k=2, F=32, act="f32", expert="relu", n_shared=1)
    w0 = wl.Workload("t", T=40, d=32, E=6, k=2, F=32, act="f32", expert="relu")
    inp = wl.make_inputs(w1, seed=22)
    inp["W2"][w1.E] = 0
    a = run_oracle(w1, inp)["y"]
    b = run_oracle(w0, dict(inp, W13=inp["W13"][: w0.E], W2=inp["W2"][: w0.E]))["y"]
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def test_shared_expert_is_never_dropped():
    """Capacity limits routed experts only; the shared expert keeps all T tokens."""
    idx = np.array([[0, 3], [0, 3], [1, 3], [0, 3]])  # expert 3 plays the shared expert
    d = orc.dispatch(idx, 4, capacity=1, D=1, capped_experts=3)
    assert d["counts_routed"].tolist() == [3, 1, 0, 4]
    assert d["counts_kept"].tolist() == [1, 1, 0, 4]
    assert d["drop_list"].tolist() == [2, 6]
    assert d["rank_offsets"].tolist() == [0, 2]


# ----------------------------------------------------------------------- drop order / padded layout
def test_gate_ordered_drop_keeps_the_largest_gates():
    """Expert 0 receives tokens 0..3 with gates .3 .9 .5 .7 and C = 2: tokens 1 and 3 stay, in token order."""
    idx = np.array([[0, 1], [0, 2], [0, 1], [0, 2]])
    gates = np.array([[0.3, 0.7], [0.9, 0.1], [0.5, 0.5], [0.7, 0.3]])
    d = orc.dispatch(idx, 3, capacity=2, gates=gates, drop_policy="gate")
    assert d["row_src"].tolist()[:2] == [2, 6]          # assignments t*k+j of tokens 1 and 3
    assert d["drop_list"].tolist() == [0, 4]             # tokens 0 and 2, expert order then token order
    assert d["counts_kept"].tolist() == [2, 2, 2]
    t = orc.dispatch(idx, 3, capacity=2)                 # token order keeps tokens 0 and 1
    assert t["row_src"].tolist()[:2] == [0, 2]


def test_gate_ordered_drop_ties_go_to_the_lower_token():
    idx = np.zeros((5, 1), np.int64)
    gates = np.array([[0.5], [0.8], [0.5], [0.8], [0.5]])
    d = orc.dispatch(idx, 1, capacity=3, gates=gates, drop_policy="gate")
    assert d["row_src"].tolist() == [0, 1, 3]            # both 0.8s, then the first 0.5
    assert d["drop_list"].tolist() == [2, 4]


def _brute_gate_dispatch(idx, gates, E, C):
    T, k = idx.shape
    kept, drops = [], []
    for e in range(E):
        mine = [(-gates[t, j], t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        chosen = set((t, j) for _, t, j in sorted(mine)[:C])
        kept += [t * k + j for _, t, j in sorted(mine, key=lambda m: m[1]) if (t, j) in chosen]
        drops += [t * k + j for _, t, j in sorted(mine, key=lambda m: m[1]) if (t, j) not in chosen]
    return kept, drops


@pytest.mark.parametrize("C", [0, 1, 2, 5, 50])
def test_gate_ordered_drop_matches_brute_force(C):
    r = rng(31)
    T, E, k = 41, 5, 2
    idx = np.stack([r.permutation(E)[:k] for _ in range(T)])
    gates = np.round(r.random((T, k)), 2)  # rounded so that some gates tie
    d = orc.dispatch(idx, E, C, gates=gates, drop_policy="gate")
    kept, drops = _brute_gate_dispatch(idx, gates, E, C)
    assert d["row_src"].tolist() == kept and d["drop_list"].tolist() == drops


def test_padded_layout_rows_and_layout_invariance():
    w = wl.Workload("t", T=60, d=16, E=4, k=2, F=24, act="f32", expert="swiglu", capacity_factor="1")
    inp = wl.make_inputs(w, seed=32)
    packed = run_oracle(w, inp)
    padded = run_oracle(wl.scaled(w, layout="padded"), inp)
    C = orc.expert_capacity(w.T, w.k, w.E, "1")
    assert padded["offsets"].tolist() == [e * C for e in range(w.E + 1)]
    for e in range(w.E):
        n = packed["counts_kept"][e]
        lo = packed["offsets"][e]
        np.testing.assert_array_equal(padded["row_src"][e * C:e * C + n], packed["row_src"][lo:lo + n])
        assert np.all(padded["row_src"][e * C + n:(e + 1) * C] == -1)
        assert np.all(padded["xperm"][e * C + n:(e + 1) * C] == 0)
    np.testing.assert_array_equal(padded["y"], packed["y"])


def test_gate_policy_equals_token_policy_without_overflow():
    w = wl.Workload("t", T=30, d=16, E=4, k=2, F=24, act="f32", expert="relu", capacity_factor="4")
    inp = wl.make_inputs(w, seed=33)
    a = run_oracle(w, inp)
    b = run_oracle(wl.scaled(w, drop_policy="gate"), inp)
    assert a["n_dropped"] == 0 and np.array_equal(a["row_src"], b["row_src"])


# ------------------------------------------------------------ group-limited routing
def _greedy_group_limited(h, k, gs, M):
    """The walk description: experts in KeepTopK order (logit desc, id asc), skipping an
    expert whose group would be the (M+1)-th distinct group."""
    order = sorted(range(len(h)), key=lambda e: (-h[e], e))
    groups, out = [], []
    for e in order:
        g = e // gs
        if g not in groups:
            if len(groups) == M:
                continue
            groups.append(g)
        out.append(e)
        if len(out) == k:
            break
    return out


@pytest.mark.parametrize("E,G,M,k", [(12, 4, 2, 3), (16, 8, 3, 4), (8, 2, 1, 2), (24, 6, 4, 8)])
def test_group_limited_topk_matches_the_greedy_walk(E, G, M, k):
    r = rng(40 + E)
    H = r.normal(size=(200, E))
    H[:20] = np.round(H[:20], 1)  # some equal logits and equal group scores
    got = orc.keep_topk_grouped(H, k, G, M)
    for t in range(H.shape[0]):
        assert got[t].tolist() == _greedy_group_limited(H[t], k, E // G, M), t


def test_group_limited_topk_hand_case():
    # groups {0,1} {2,3} {4,5} {6,7}; scores 0.9, 0.8, 0.85, 0.3 -> keep groups 0 and 2
    H = np.array([[0.9, 0.1, 0.8, 0.7, 0.85, 0.0, 0.2, 0.3]])
    assert orc.keep_topk_grouped(H, 3, 4, 2).tolist() == [[0, 4, 1]]
    assert orc.keep_topk(H, 3).tolist() == [[0, 4, 2]]
    # equal scores keep the lower groups
    assert orc.keep_topk_grouped(np.zeros((1, 8)), 3, 4, 2).tolist() == [[0, 1, 2]]


def test_group_limited_topk_invariants():
    r = rng(41)
    E, G, M, k = 32, 8, 3, 6
    H = r.normal(size=(300, E))
    idx = orc.keep_topk_grouped(H, k, G, M)
    full = orc.keep_topk(H, k)
    for t in range(H.shape[0]):
        groups = set((idx[t] // (E // G)).tolist())
        assert len(groups) <= M
        if len(set((full[t] // (E // G)).tolist())) <= M:  # the limit does not bind
            assert idx[t].tolist() == full[t].tolist()
    assert np.array_equal(orc.keep_topk_grouped(H, k, G, G), full)  # M = G: no limit


def test_group_tie_flags():
    H = np.array([[1.0, 0.0, 0.5, 0.0, 0.5 * (1 + 1e-8), 0.0],
                  [1.0, 0.0, 0.5, 0.0, 0.4, 0.0]])
    assert orc.group_tie_flags(H, 3, 2).tolist() == [True, False]
    assert not orc.group_tie_flags(H, 3, 3).any()


def test_forward_with_group_limit_keeps_at_most_m_groups():
    w = wl.Workload("t", T=64, d=32, E=16, k=4, F=16, act="f32", expert="relu", D=4)
    inp = wl.make_inputs(w, seed=42)
    res = orc.moe_forward(f64(inp["x"]), f64(inp["Wg"]), w.k, expert_fn(w.expert, inp["W13"], inp["W2"], w.F),
                          n_groups=4, topk_groups=2)
    assert all(len(set((row // 4).tolist())) <= 2 for row in res["idx"])
    np.testing.assert_allclose(res["G"].sum(axis=1), 1.0, rtol=1e-12)


# ------------------------------------------------------------ deduplicated dispatch
def test_dedup_brute_force_expectation_is_the_exact_closed_form():
    # every k-subset of E experts as one token: the mean number of ranks touched is
    # D (1 - C(E - E/D, k) / C(E, k)) exactly
    E, D = 8, 4
    for k in (1, 2, 3, 5):
        idx = np.array(list(itertools.combinations(range(E), k)))
        d = orc.dispatch(idx, E)
        s = orc.dedup_send(idx, d["pos"], E, D)
        exact = Fraction(D) * (1 - Fraction(math.comb(E - E // D, k), math.comb(E, k)))
        assert Fraction(s["n_send"], len(idx)) == exact


def test_dedup_closed_form_tends_to_the_pages_with_replacement_figure():
    # with many experts per rank, drawing k distinct experts is close to k independent
    # uniform rank picks: D (1 - (1 - 1/D)^k) ~ 5.25 for D = k = 8. Distinct experts
    # touch slightly more ranks (5.29): a second pick avoids the first expert.
    E, D, k = 256, 8, 8
    exact = D * (1 - math.comb(E - E // D, k) / math.comb(E, k))
    with_replacement = D * (1 - (1 - 1 / D) ** k)
    assert with_replacement < exact < with_replacement * 1.01
    assert round(D * (1 - (1 - 1 / D) ** k), 2) == 5.25 and round((D - 1) * (1 - (1 - 1 / D) ** k), 1) == 4.6


def test_dedup_layout_and_fan_out():
    r = rng(43)
    T, E, k, D = 90, 16, 4, 4
    idx = np.stack([r.permutation(E)[:k] for _ in range(T)])
    d = orc.dispatch(idx, E, 20, D)  # capacity 20: some drops
    assert d["n_dropped"] > 0
    s = orc.dedup_send(idx, d["pos"], E, D)
    # rows are rank-major, token order inside a rank, one per (token, rank) pair with a kept assignment
    pairs = sorted({(int(e) // (E // D), t) for t in range(T) for j, e in enumerate(idx[t])
                    if d["pos"][t * k + j] >= 0})
    assert s["send_src"].tolist() == [t * D + rr for rr, t in pairs]
    assert s["send_counts"].tolist() == [sum(1 for rr, _ in pairs if rr == q) for q in range(D)]
    for a in range(T * k):
        t, e = a // k, idx[a // k, a % k]
        if d["pos"][a] >= 0:
            assert s["send_src"][s["fan_src"][a]] == t * D + e // (E // D)
        else:
            assert s["fan_src"][a] == -1
    # k = 1: one row per token; D = 1: one row per token with any kept assignment
    one = orc.dedup_send(idx[:, :1], orc.dispatch(idx[:, :1], E)["pos"], E, D)
    assert one["n_send"] == T
    assert orc.dedup_send(idx, d["pos"], E, 1)["n_send"] == int((d["pos"].reshape(T, k) >= 0).any(axis=1).sum())


def test_dedup_skips_shared_experts():
    T, E, S = 10, 8, 1
    idx = np.concatenate([np.tile([0, 5], (T, 1)), np.full((T, S), E)], axis=1)
    d = orc.dispatch(idx, E + S, None, 2, capped_experts=E)
    s = orc.dedup_send(idx, d["pos"], E, 2)
    assert s["n_send"] == 2 * T and np.all(s["fan_src"].reshape(T, 3)[:, 2] == -1)


# ------------------------------------------------------------ FP8 dispatch
def test_e4m3_table():
    v = orc.e4m3_values()
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.sum(~np.isnan(v)) == 254
    assert v[0x7E] == 448.0 and v[0x38] == 1.0 and v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert np.array_equal(v[0x80:0xFF], -v[0x00:0x7F]) and np.all(np.diff(v[:0x7F]) > 0)


def test_e4m3_rounding_matches_torch_float8():
    r = rng(50)
    x = r.normal(size=50000) * r.choice([1e-3, 0.05, 1.0, 30.0, 300.0], 50000)
    x = x[np.abs(x) <= 448].astype(np.float32).astype(np.float64)
    ref = torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc._e4m3_round(x), ref)


def test_e4m3_rounding_hand_cases():
    cases = [(1.0625, 0x38),          # halfway between 1.0 (even) and 1.125
             (1.1875, 0x3A),          # halfway between 1.125 and 1.25 (even)
             (2.0 ** -10, 0x00),      # halfway between 0 and the smallest subnormal: +0
             (-(2.0 ** -11), 0x80),   # rounds to zero, keeps its sign
             (0.0, 0x00), (-0.0, 0x80), (448.0, 0x7E), (-448.0, 0xFE), (3.3, 0x45)]
    for x, code in cases:
        assert int(orc._e4m3_round(np.array([x]))[0]) == code, x


def test_fp8_block_scales_and_error_bound():
    x = np.zeros((4, 200))
    x[0, 0], x[1, 5], x[2, 7] = 448.0, 449.0, 1.0    # first blocks: s = 0, 1, -8
    x[3, 150] = -3.0                                 # ragged second block (72 elements)
    q = orc.quantize_fp8_blocks(x)
    assert q["exps"].tolist() == [[0, 0], [1, 0], [-8, 0], [0, -7]]
    assert q["deq"][1, 5] == 448.0 and q["deq"][3, 150] == -3.0 and not q["deq"][0, 1:].any()
    r = rng(51)
    x = r.normal(size=(16, 384)) * np.exp(r.normal(size=(16, 1)) * 3)
    q = orc.quantize_fp8_blocks(x)
    s = np.repeat(q["exps"], 128, axis=1)
    amax = np.abs(x).reshape(16, 3, 128).max(axis=2)
    assert np.all(amax / 2.0 ** q["exps"] <= 448) and np.all(amax / 2.0 ** (q["exps"] - 1) > 448)  # smallest s
    err = np.abs(q["deq"] - x)
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** (s - 10)))
    # dequantized rows are fixed points (their codes may differ: a block's amax can round
    # down to a value that takes a smaller scale)
    assert np.array_equal(orc.quantize_fp8_blocks(q["deq"])["deq"], q["deq"])


def test_fp8_forward_sends_the_dequantized_rows():
    w = wl.Workload("t", T=40, d=256, E=4, k=1, F=0, act="bf16", expert="identity")
    inp = wl.make_inputs(w, seed=52)
    res = orc.moe_forward(f64(inp["x"]), f64(inp["Wg"]), 1, lambda e, X: X, dispatch_dtype="fp8")
    np.testing.assert_array_equal(res["y"], orc.quantize_fp8_blocks(f64(inp["x"]))["deq"])


def test_fp8_rows_are_the_block_rule_with_one_block_per_row():
    r = rng(53)
    x = r.normal(size=(40, 300)) * np.exp(r.normal(size=(40, 1)) * 4)
    x[3] = 0.0
    x[5] = -0.0
    x[7, 11] = 449.0
    x[8, :] = 2.0 ** -140  # far below e4m3's range: a large negative scale exponent
    q = orc.quantize_fp8_rows(x, chunk=7)
    b = orc.quantize_fp8_blocks(x, block=300)
    assert np.array_equal(q["codes"], b["codes"]) and np.array_equal(q["exps"], b["exps"][:, 0])
    assert np.array_equal(q["deq"], b["deq"])
    assert q["exps"][3] == 0 and not q["deq"][3].any() and np.all(q["codes"][5] == 0x80)
    assert q["exps"][8] == -148 and np.all(q["deq"][8] == 2.0 ** -140)  # 2^-140 / 2^-148 = 256 <= 448 < 512
    # cross-check of the codes against torch's float8 conversion of x / 2^s
    ref = torch.tensor(np.ldexp(x, -q["exps"][:, None]), dtype=torch.float64).to(torch.float32)
    assert np.array_equal(q["codes"], ref.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_fp8_gemm_forward_quantizes_every_kept_row_once_per_token():
    w = wl.Workload("t", T=40, d=256, E=4, k=1, F=0, act="bf16", expert="identity", n_shared=1)
    inp = wl.make_inputs(w, seed=54)
    x = f64(inp["x"])
    res = orc.moe_forward(x, f64(inp["Wg"]), 1, lambda e, X: X, n_shared=1, dispatch_dtype="fp8_gemm")
    # one routed expert (gate 1) plus the shared one (gate 1), both fed the row-quantized token
    np.testing.assert_array_equal(res["y"], 2 * orc.quantize_fp8_rows(x)["deq"])


def test_fp8_expert_equals_the_plain_expert_on_e4m3_exact_weights():
    """Weights whose rows are e4m3 values times one power of two per row (with a
    full-range value in each row, so the row scale is that power) quantize to
    themselves: the FP8 up projection must then be the plain expert exactly."""
    from oracle.packed import expert_fn
    r = rng(55)
    E, d, F = 2, 64, 32
    vals = orc.e4m3_values()[:0x7F]
    codes = r.integers(0, 0x7F, size=(E, 2 * F, d))
    W13 = vals[codes] * np.where(r.random((E, 2 * F, d)) < 0.5, -1, 1)
    W13[:, :, 0] = 448.0
    W13 = W13 * np.ldexp(1.0, r.integers(-12, -4, size=(E, 2 * F, 1)))
    W2 = r.normal(size=(E, d, F))
    X = r.normal(size=(5, d))
    plain = expert_fn("swiglu", W13, W2, F)
    fp8 = expert_fn("swiglu", W13, W2, F, fp8_up=True)
    for e in range(E):
        np.testing.assert_array_equal(fp8(e, X), plain(e, X))
    # a weight that is not e4m3-exact changes the result
    W13[0, 0, 1] = 448.0 * 1.01 * 2.0 ** -12
    assert not np.array_equal(expert_fn("swiglu", W13, W2, F, fp8_up=True)(0, X), plain(0, X))



def test_fp8_hidden_rounds_to_bf16_first():
    """h is stored in bf16 before it is quantized: a value just above an e4m3 midpoint
    that bf16 rounds onto the midpoint then ties to the even e4m3 code."""
    h = np.array([[448.0, 1.0625 + 2.0 ** -12, 1.1875 + 2.0 ** -12, -3.0]])  # row scale 2^0
    got = orc.fp8_hidden(h)
    # direct e4m3 rounding would give 1.125 and 1.25 for the two middle values
    assert got.tolist() == [[448.0, 1.0, 1.25, -3.0]]
    assert orc.quantize_fp8_rows(h)["deq"].tolist() == [[448.0, 1.125, 1.25, -3.0]]
    # a row whose largest value is 0.5 takes the scale 2^-9 and keeps e4m3-exact values
    h = np.array([[0.5, 0.25 * 1.125, -0.0009765625]])
    assert np.array_equal(orc.fp8_hidden(h), h)


def test_fp8_down_projection_equals_the_plain_expert_on_exact_values():
    """ReLU experts with one-hot token rows, so h is a set of rows of W1^T: with W1, W2
    e4m3 values times one power of two per row (and a full-range value per row) every
    quantization is exact and the FP8 expert must equal the plain one."""
    from oracle.packed import expert_fn
    r = rng(56)
    E, d, F = 2, 32, 48
    vals = orc.e4m3_values()[:0x7F]

    def exact_rows(n, m, lo, hi):
        w = vals[r.integers(0, 0x7F, size=(E, n, m))] * np.where(r.random((E, n, m)) < 0.5, -1, 1)
        w[:, :, 0] = 448.0
        return w * np.ldexp(1.0, r.integers(lo, hi, size=(E, n, 1)))

    W1 = np.abs(exact_rows(F, d, -10, -6))  # [E, F, d], rows = output channels, >= 0 so relu keeps h
    W2 = exact_rows(d, F, -12, -8)          # [E, d, F]
    # token rows one-hot on column 0: h[f] = W1[e, f, 0] = 448 * 2^s_f, s_f within 4 of
    # each other, so h is bf16-exact and e4m3-exact under its row scale
    X = np.zeros((4, d))
    X[:, 0] = 1.0
    plain = expert_fn("relu", W1, W2, F)
    fp8 = expert_fn("relu", W1, W2, F, fp8_up=True, fp8_h=True)
    for e in range(E):
        np.testing.assert_array_equal(fp8(e, X), plain(e, X))
    # a token value that is not e4m3-exact changes the result
    X2 = np.zeros((1, d))
    X2[0, 0] = 1.0
    X2[0, 1] = 1.0 + 2.0 ** -20
    assert not np.array_equal(fp8(0, X2), plain(0, X2))
