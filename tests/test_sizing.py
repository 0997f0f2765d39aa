"""Host-side byte/parameter helpers reproduce the worked numbers the pages print."""
import json
import os

import pytest

from routing_dispatch_combine_moe_b300 import sizing as sz

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_numbers.json")))
MB, GB = 1e6, 1e9


def value(name):
    g = GOLD[name]
    i = g["inputs"]
    if name == "assignments_dsv3_rank":
        return sz.assignments(i["T"], i["k"])
    if name == "mean_per_expert_dsv3":
        return sz.assignments(i["T"], i["k"]) / i["E"]
    if name == "dispatch_mb_per_direction_dsv3":
        return sz.dispatch_bytes_per_direction(i["T"], i["k"], i["d"], i["bytes"]) / MB
    if name in ("dispatch_mb_ep64", "dispatch_mb_8nodes"):
        return sz.dispatch_bytes_per_direction(i["T"], i["k"], i["d"], i["bytes"], D=i["D"]) / MB
    if name == "dispatch_ms_8nodes_50gbs":
        return i["MB"] / i["GBs"]
    if name == "straggler_gb":
        return i["MB"] * (1 + i["imbalance"]) / 1000
    if name == "params_per_gated_expert_dsv3":
        return sz.gated_expert_params(i["d"], i["F"])
    if name == "routed_expert_params_dsv3_58_layers":
        return sz.gated_expert_params(i["d"], i["F"]) * i["E"] * i["layers"]
    if name == "params_per_rank_ep64":
        return sz.gated_expert_params(i["d"], i["F"]) * i["experts_per_rank"] * i["layers"]
    if name == "dense4_expert_params_d4096":
        return sz.dense4_expert_params(i["d"])
    if name == "dense4_expert_params_64_experts":
        return sz.dense4_expert_params(i["d"]) * i["E"]
    if name == "dense4_expert_params_per_device_D8":
        return sz.dense4_expert_params(i["d"]) * i["E"] / i["D"]
    if name == "experts_per_device_E64_D8":
        return i["E"] // i["D"]
    if name == "decode_vectors":
        return sz.assignments(i["T"], i["k"])
    if name in ("decode_dispatch_mb_fp8", "decode_combine_mb_bf16"):
        return sz.dispatch_bytes_per_direction(i["T"], i["k"], i["d"], i["bytes"]) / MB
    if name == "decode_dispatch_us_50gbs":
        return sz.dispatch_bytes_per_direction(i["T"], i["k"], i["d"], i["bytes"]) / (i["GBs"] * GB) * 1e6
    if name == "expected_nodes_touched_k8_n8":
        return sz.expected_nodes_touched(i["k"], i["n"])
    if name == "expected_remote_nodes_k8_n8":
        return sz.expected_remote_nodes(i["k"], i["n"])
    if name == "home_node_touch_probability":
        return 1 - (1 - 1 / i["n"]) ** i["k"]
    if name == "dedup_expected_mb":
        return i["T"] * sz.expected_remote_nodes(i["k"], i["n"]) * i["d"] * i["bytes"] / MB
    if name == "node_limited_3_remote_mb":
        return i["T"] * i["remote_nodes"] * i["d"] * i["bytes"] / MB
    if name == "strict_4_remote_copies":
        return i["T"] * i["remote_nodes"]
    if name == "strict_4_remote_mb":
        return i["T"] * i["remote_nodes"] * i["d"] * i["bytes"] / MB
    if name == "whole_model_gb":
        return i["MB"] * i["layers"] * i["directions"] / 1000
    if name == "capacity_zipf_workload":
        return sz.capacity(i["T"], i["k"], i["E"], i["f"])
    raise KeyError(name)


@pytest.mark.parametrize("name", [k for k in GOLD if not k.startswith("_")])
def test_worked_number(name):
    g = GOLD[name]
    got = value(name)
    if g["rel_tol"] == 0:
        assert got == g["printed"]
    else:
        assert got == pytest.approx(g["printed"], rel=g["rel_tol"])


def test_dispatch_bytes_independent_of_E_and_layer_is_twice():
    a = sz.dispatch_bytes_per_direction(4096, 8, 7168, 2, D=8)
    assert sz.layer_comm_bytes(4096, 8, 7168, 2, D=8) == 2 * a


def test_capacity_exact_rational():
    assert sz.capacity(10, 1, 3, "1") == 4
    assert sz.capacity(10, 1, 3, "0.9") == 3
    assert sz.capacity(10, 1, 3, "0.91") == 4
    assert sz.capacity(16, 2, 8, "1.0", min_capacity=6) == 6
    assert sz.capacity(16, 2, 8, None) is None
    assert sz.capacity_fraction("1.25") == (5, 4)


def test_imbalance_ratio_definition():
    assert sz.imbalance_ratio([1, 1, 1, 5]) == pytest.approx((5 - 2) / 2)
    assert sz.imbalance_ratio([3, 3, 3]) == 0.0


def test_remote_dispatch_bytes():
    assert sz.remote_dispatch_bytes([0, 10, 25, 40], d=4, elem_bytes=2) == (15 + 15) * 4 * 2
