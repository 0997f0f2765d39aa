"""The split of the expert GEMM's last partial wave over k.

When the swapped-pair down projection's tiles leave the last wave of SM pairs at most
half busy, each tile of that wave is cut into ranges of k-blocks run on otherwise idle
pairs, and the range that finishes last sums the ranges' fp32 partials in range order.
The cases below give every expert 300 rows (two token tiles) and d = 1280 (five
feature tiles): 80 tiles for the 74 pairs of a B300, so the last wave's 6 tiles are cut
into 4 ranges each. MOE_GEMM_SPLITK=0 (read once per process) turns the split off, so
each case runs in two child processes, split on and off. Both must match the oracle's
experts within the stated tolerance; the two outputs must differ (the split ran: the
sums are associated differently) by no more than two fp32 summations of the same n
products can: |s1 - s2| <= 2 (n - 1) u sum_i |x_i|, u = 2^-24 (the recursive-summation
bound, Higham, "Accuracy and Stability of Numerical Algorithms", section 4.2), with
sum_i |x_i| = |h| . |w| taken from the h each run stored and the bf16 W2. A range
dropped or counted twice moves an element by a share of the whole sum, hundreds of
times that bound.
"""
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
from routing_dispatch_combine_moe_b300 import workloads as wl, abi
from tests._gpu import StageBuffers, check_ffn
w = wl.scaled(wl.WORKLOADS[{base!r}], T=1536, d=1280, F=2048, **{changes!r})
inp = wl.make_inputs(w, 3, device="cuda")
cfg = abi.config_for(w)
b = StageBuffers(w, cfg)
counts = torch.full((w.n_experts,), 300, dtype=torch.int64)
g = torch.Generator().manual_seed(11)
xperm = torch.randn(int(counts.sum()), w.d, generator=g).to(w.torch_act).cuda()
err = check_ffn(w, inp, b, dict(counts=counts, xperm=xperm))
assert b.ffn_status() == 0
n = int(counts.sum())
np.save({path!r} + ".out.npy", b.out[:n].float().cpu().numpy())
# sum_i |h_i w_i| of every output and the number of products (hi and lo both meet w)
h = b.h[:n].float().cpu().numpy().astype(np.float64)
if w.precision == "split_h":
    h4 = h.reshape(n, w.F // 64, 2, 64)
    habs, nprod = (np.abs(h4[:, :, 0, :]) + np.abs(h4[:, :, 1, :])).reshape(n, w.F), 2 * w.F
else:
    habs, nprod = np.abs(h), w.F
W2 = np.abs(inp["W2"].float().cpu().numpy().astype(np.float64))
A = np.concatenate([habs[300 * e:300 * (e + 1)] @ W2[e].T for e in range(w.n_experts)])
np.save({path!r} + ".abs.npy", A)
print("nprod", nprod)
print("ffn_err/rms", err)
print("ok")
"""

CASES = {
    "f32_out": ("mixtral_bf16", {}),
    "split_h": ("mixtral_bf16", {"precision": "split_h"}),
    "bf16_out": ("mixtral_bf16", {"precision": "bf16"}),
    "fp8_h": ("mixtral_fp8_experts", {}),
}


def _run(case, split, path):
    base, changes = CASES[case]
    env = dict(os.environ, MOE_GEMM_SPLITK=split)
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT, base=base, changes=changes, path=path)],
                       env=env, capture_output=True, text=True, timeout=900)
    print(r.stdout[-2000:])
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-3000:]
    nprod = int(r.stdout.split("nprod")[1].split()[0])
    return np.load(path + ".out.npy").astype(np.float64), np.load(path + ".abs.npy"), nprod


@pytest.mark.parametrize("case", list(CASES))
def test_split_k_tail_matches_whole_k_tiles(case):
    with tempfile.TemporaryDirectory() as tmp:
        on, abs_on, nprod = _run(case, "1", os.path.join(tmp, "on"))
        off, abs_off, _ = _run(case, "0", os.path.join(tmp, "off"))
    assert on.shape == off.shape and np.isfinite(on).all() and np.isfinite(off).all()
    # both runs computed the same h (the up projection is never split)
    assert np.array_equal(abs_on, abs_off)
    rms = float(np.sqrt(np.mean(off ** 2)))
    diff = np.abs(on - off)
    bound = 2 * (nprod - 1) * 2.0 ** -24 * abs_on
    if case == "fp8_h":
        bound *= 2  # the GEMM's e4m3 h and W2 are within 2^-4 of the bf16 ones (normal codes)
    if case == "bf16_out":
        # then one rounding to bf16 each: up to one bf16 ulp (2^-7 of the larger) apart
        bound = bound + np.maximum(np.abs(on), np.abs(off)) * 2.0 ** -7
    print(f"{case}: split on/off max|diff|/rms = {diff.max() / rms:.3e}, differing elements "
          f"{(diff > 0).mean():.4f}, max diff/bound {(diff / np.maximum(bound, 1e-300)).max():.3e}")
    assert (diff > 0).any(), "the split did not run: outputs are bit-identical"
    assert np.all(diff <= bound), f"{case}: split on/off differ beyond the summation-order bound"

