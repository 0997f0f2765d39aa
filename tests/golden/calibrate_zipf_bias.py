"""Find the Zipf bias scale that makes the hot expert draw 40% of the assignments.

The imbalanced workload (T=8192, d=2048, E=64, k=2, Zipf s=1.2) biases the router
logits by b_e = -lambda * s * ln(rank_e). This script bisects lambda on the
oracle's routing of the seed-0 router inputs until the hot expert's share of the
T*k assignments is 40%, and writes the result to zipf_bias_lambda.json beside it.
It calls only the oracle and the seeded input generator.

    python tests/golden/calibrate_zipf_bias.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import moe_oracle as orc  # noqa: E402
from routing_dispatch_combine_moe_b300 import workloads as wl  # noqa: E402


def hot_share(lam: float, seed: int = 0) -> float:
    w = wl.WORKLOADS["zipf_cf125"]
    x, Wg, _ = wl.make_router_inputs(w, seed)
    bias = wl.zipf_bias(w.E, w.zipf_s, seed, lam=lam)
    H = orc.router_logits(x.float().numpy(), Wg.numpy(), bias.numpy())
    idx = orc.keep_topk(H, w.k)
    counts = np.bincount(idx.ravel(), minlength=w.E)
    return counts.max() / idx.size


def main():
    lo, hi = 0.0, 4.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if hot_share(mid) < 0.40:
            lo = mid
        else:
            hi = mid
    lam = round(0.5 * (lo + hi), 6)
    share = hot_share(lam)
    out = {"lambda": lam, "hot_share_seed0": share, "target": 0.40,
           "workload": "zipf_cf125", "seed": 0}
    with open(os.path.join(HERE, "zipf_bias_lambda.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
