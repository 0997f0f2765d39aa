"""moe_dispatch_static: the dispatch for callers that cannot give the library device
memory for scratch (a serving loop that must not allocate once it runs, or a plugin
whose host framework owns every device buffer). Its scratch is one array built into
the library, so two calls in a row must each match the workspace-based moe_dispatch
bit for bit, with nothing left over from the previous call.

This file runs last in the suite (pytest collects files by name), and passes both on
its own in a fresh process and after the other tests."""
import numpy as np
import pytest
import torch

from routing_dispatch_combine_moe_b300 import abi
from routing_dispatch_combine_moe_b300 import workloads as wl
from tests._gpu import StageBuffers, cpu

pytestmark = pytest.mark.gpu

FIELDS = ["counts_routed", "counts_kept", "offsets", "rank_offsets", "pos", "n_dropped"]


def _run_both(w, seed):
    inp = wl.make_inputs(w, seed, device="cuda")
    cfg = abi.config_for(w)
    ref = StageBuffers(w, cfg)
    ref.route(inp)
    ref.dispatch(inp)
    got = StageBuffers(w, cfg)
    abi.moe_dispatch_static(cfg, inp["x"], ref.topk_idx, got.dmap(), got.xperm, topk_gate=ref.topk_gate)
    torch.cuda.synchronize()
    for f in FIELDS:
        assert torch.equal(getattr(got, f), getattr(ref, f)), f
    rows = ref.rows if w.layout == "padded" else int(cpu(ref.offsets)[-1])
    nd = int(cpu(ref.n_dropped)[0])
    assert torch.equal(got.row_src[:rows], ref.row_src[:rows])
    assert torch.equal(got.drop_list[:nd], ref.drop_list[:nd])
    assert torch.equal(got.xperm[:rows], ref.xperm[:rows])
    return rows, nd


def test_static_scratch_dispatch_matches_workspace_dispatch_twice():
    # first call: DeepSeek-V3 routing shape; second call: a different shape with
    # drops, so stale scratch from the first call would show up
    a = _run_both(wl.scaled(wl.WORKLOADS["dsv3_route_only"], T=2048), seed=11)
    b = _run_both(wl.Workload("cap", T=3000, d=256, E=64, k=2, F=0, act="bf16", expert="identity",
                              capacity_factor="1", zipf_s=1.2, D=4), seed=12)
    assert a[0] == 2048 * 8 and b[1] > 0


def test_static_scratch_gate_drops_into_padded_rows():
    # the gate drop policy uses the extra per-expert list in the static array
    _, nd = _run_both(wl.Workload("gate_pad", T=3000, d=256, E=64, k=2, F=0, act="bf16", expert="identity",
                                  capacity_factor="1", zipf_s=1.2, D=4, drop_policy="gate", layout="padded"),
                      seed=13)
    assert nd > 0


def test_static_scratch_rejects_configs_beyond_its_size():
    cfg = abi.make_config(T=1 << 20, d=64, E=256, k=8, expert="identity")
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    m = abi.dispatch_map(*([x] * 8))
    with pytest.raises(abi.MoeError) as e:
        abi.moe_dispatch_static(cfg, x, x, m, x)
    assert e.value.code == abi.MOE_ERR_WORKSPACE
