"""The five synthetic MoE-layer workloads and their seeded input generator.

This module draws random inputs and nothing else: it holds none of the layer's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Recipe (every config): x ~ N(0, 1); router weight W_g ~ N(0, 1/d), fp32; expert
weights ~ N(0, 1/fan_in). Values are drawn in fp32 and then cast to the activation
dtype. The router-side inputs (x, W_g, the per-expert bias) come from a CPU
generator so that they are the same whichever device receives them; expert
weights come from a generator on the target device (seeded from the same seed),
because the largest workload holds 22.5 GB of them.

Expert weight layout (the usual "linear layer" orientation, K-major for the GEMMs):

* ``W13`` [E, R, d]: for SwiGLU R = 2F, rows [0, F) are W_gate^T and rows [F, 2F)
  are W_up^T; for ReLU R = F and the rows are W_1^T.
* ``W2``  [E, d, F]: W_down^T (ReLU: W_2^T).

So the math-layout matrices are W_gate[e] = W13[e, :F].T (d x F) and
W_down[e] = W2[e].T (F x d).

The imbalanced workload adds a per-expert router bias b_e = -lambda * s * ln(rank_e)
with Zipf exponent s = 1.2 over a seeded random ranking of the experts (rank 1 is
the hot expert, whose bias is 0), i.e. b_e = lambda * ln(p_rank / p_1) for Zipf
probabilities p_r proportional to r^-s. lambda = ZIPF_LAMBDA was found by bisection
on the oracle's routing of seed 0 so that the hot expert draws 40% of the T*k
assignments (tests/golden/calibrate_zipf_bias.py reproduces it).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

ZIPF_LAMBDA = 1.059709  # hot expert draws 40.0% of assignments on seed 0


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    act: str  # "f32" | "bf16"
    expert: str  # "relu" | "swiglu" | "identity"
    capacity_factor: str | None = None  # exact decimal string; None = dropless
    min_capacity: int = 0
    D: int = 1  # virtual expert-parallel ranks the dispatch is laid out for
    zipf_s: float | None = None
    # bf16 experts: "bf16" (h and expert outputs in bf16), "f32_out" (expert outputs in
    # fp32), "split_h" (h as a bf16 hi/lo pair too) or "fp8_h" (with dispatch_dtype
    # "fp8_gemm": h quantized to e4m3 per row, the down projection on e4m3); see the
    # library header.
    precision: str = "f32_out"
    n_shared: int = 0  # shared experts (ids E .. E+n_shared-1) every token also uses, gate 1
    drop_policy: str = "token"  # overflow dropped in token order, or "gate": lowest gates first
    layout: str = "packed"      # "packed" rows, or "padded": a fixed segment of C rows per expert
    n_groups: int = 0           # expert groups for group-limited routing (with topk_groups)
    topk_groups: int = 0        # 0 < M < n_groups: each token keeps experts of at most M groups
    dedup: bool = False         # send each token once per virtual rank, then fan out
    dispatch_dtype: str = "act"  # "fp8": routed rows travel as e4m3 with per-128 block scales;
    # "fp8_gemm": every row as row-scaled e4m3, fed to an FP8 up projection (e4m3 W13)
    note: str = field(default="", compare=False)

    @property
    def torch_act(self) -> torch.dtype:
        return torch.float32 if self.act == "f32" else torch.bfloat16

    @property
    def act_bytes(self) -> int:
        return 4 if self.act == "f32" else 2

    @property
    def n_experts(self) -> int:
        """Routed plus shared experts (the expert weights hold this many)."""
        return self.E + self.n_shared

    @property
    def slots(self) -> int:
        """Experts each token visits: k routed plus the shared ones."""
        return self.k + self.n_shared

    @property
    def w13_rows(self) -> int:
        return 2 * self.F if self.expert == "swiglu" else self.F


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_f32", T=256, d=128, E=8, k=2, F=256, act="f32", expert="relu",
                 note="tiny fp32 layer, ReLU experts, dropless"),
        Workload("mixtral_bf16", T=2048, d=4096, E=8, k=2, F=14336, act="bf16",
                 expert="swiglu", note="Mixtral-shaped layer, SwiGLU experts, dropless"),
        Workload("dsv3_route_only", T=4096, d=7168, E=256, k=8, F=0, act="bf16",
                 expert="identity", D=8,
                 note="DeepSeek-V3-shaped routing+dispatch+combine, identity experts, "
                      "8 virtual ranks of 32 experts"),
        Workload("zipf_cf125", T=8192, d=2048, E=64, k=2, F=1408, act="bf16",
                 expert="swiglu", capacity_factor="1.25", zipf_s=1.2, precision="split_h",
                 note="Zipf(1.2)-biased router, capacity factor 1.25, token-order drops; the drops "
                      "shrink rms(y), so h is carried as a bf16 hi/lo pair"),
        Workload("dsv3_full", T=4096, d=7168, E=256, k=8, F=2048, act="bf16",
                 expert="swiglu", note="DeepSeek-V3-shaped full layer, 22.5 GB of experts"),
        Workload("dsv3_decode", T=128, d=7168, E=256, k=8, F=2048, act="bf16", expert="swiglu",
                 n_shared=1, D=8,
                 note="decode-shaped DeepSeek-V3 layer: 128 tokens, 8 routed experts plus the shared "
                      "expert per token (9 vectors each), 8 virtual ranks"),
        Workload("dsv3_grouped_dedup", T=4096, d=7168, E=256, k=8, F=0, act="bf16", expert="identity", D=8,
                 n_groups=8, topk_groups=4, dedup=True,
                 note="DeepSeek-V3 routing shape with each token limited to 4 of 8 expert groups (one "
                      "group per virtual rank) and the send buffer deduplicated per rank"),
        Workload("mixtral_fp8_dispatch", T=2048, d=4096, E=8, k=2, F=14336, act="bf16", expert="swiglu",
                 dispatch_dtype="fp8",
                 note="the Mixtral-shaped layer with its dispatched rows sent as e4m3 codes and "
                      "per-128 power-of-two scales"),
            Workload("mixtral_fp8_gemm", T=2048, d=4096, E=8, k=2, F=14336, act="bf16", expert="swiglu",
                 dispatch_dtype="fp8_gemm",
                 note="the Mixtral-shaped layer with its dispatched rows as row-scaled e4m3 codes fed as "
                      "they are to an FP8 up projection (e4m3 W13, one scale per output channel); h and the "
                      "down projection stay bf16"),
        Workload("dsv3_decode_fp8_gemm", T=128, d=7168, E=256, k=8, F=2048, act="bf16", expert="swiglu",
                 n_shared=1, D=8, dispatch_dtype="fp8_gemm",
                 note="the decode-shaped DeepSeek-V3 layer with FP8 rows and e4m3 up-projection weights: "
                      "the weight stream of the up projection halves"),
        Workload("mixtral_fp8_experts", T=2048, d=4096, E=8, k=2, F=14336, act="bf16", expert="swiglu",
                 dispatch_dtype="fp8_gemm", precision="fp8_h",
                 note="the Mixtral-shaped layer with both expert projections on e4m3: FP8 rows and W13 for "
                      "the up projection, h quantized per row and e4m3 W2 for the down projection"),
        Workload("dsv3_full_fp8_gemm", T=4096, d=7168, E=256, k=8, F=2048, act="bf16", expert="swiglu",
                 dispatch_dtype="fp8_gemm",
                 note="the DeepSeek-V3-shaped full layer with FP8 rows and e4m3 up-projection weights "
                      "(15.0 GB of bf16 W13 become 7.5 GB)"),
        Workload("dsv3_grouped_dedup_fp8", T=4096, d=7168, E=256, k=8, F=0, act="bf16", expert="identity", D=8,
                 n_groups=8, topk_groups=4, dedup=True, dispatch_dtype="fp8",
                 note="the group-limited, deduplicated DeepSeek-V3 routing shape with the send rows as e4m3 "
                      "codes and per-128 power-of-two scales, dequantized by the receiving side's fan-out"),
        Workload("dsv3_full_fp8_gemm_dedup", T=4096, d=7168, E=256, k=8, F=2048, act="bf16", expert="swiglu",
                 D=8, n_groups=8, topk_groups=4, dedup=True, dispatch_dtype="fp8_gemm",
                 note="the DeepSeek-V3-shaped full layer, group-limited to 4 of 8 groups, with the send rows "
                      "deduplicated per rank and sent as row-scaled e4m3 codes that the receiving side hands "
                      "to the FP8 up projection as they are"),
        Workload("dsv3_e32_slice", T=512, d=7168, E=32, k=8, F=2048, act="bf16", expert="swiglu",
                 note="an eighth of the DeepSeek-V3-shaped layer: the same d, F and k and the same 128 rows per "
                      "expert on average, with 32 experts (2.8 GB of weights), small enough for counter captures"),
    ]
}

# Workload order as they are listed: small parity case first, headline second.
WORKLOAD_ORDER = ["tiny_f32", "mixtral_bf16", "dsv3_route_only", "zipf_cf125", "dsv3_full", "dsv3_decode",
                  "dsv3_grouped_dedup", "mixtral_fp8_dispatch", "mixtral_fp8_gemm", "dsv3_decode_fp8_gemm",
                  "dsv3_full_fp8_gemm", "mixtral_fp8_experts", "dsv3_grouped_dedup_fp8", "dsv3_full_fp8_gemm_dedup",
                  "dsv3_e32_slice"]


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some sizes changed (for reduced-size parity cases)."""
    fields = dict(w.__dict__)
    fields.update(changes)
    fields.setdefault("name", w.name)
    return Workload(**fields)


def zipf_bias(E: int, s: float, seed: int, lam: float | None = None) -> torch.Tensor:
    """Per-expert router bias b_e = -lam * s * ln(rank_e) over a seeded ranking."""
    lam = ZIPF_LAMBDA if lam is None else lam
    g = torch.Generator().manual_seed(seed * 7919 + 17)
    rank = torch.randperm(E, generator=g) + 1  # rank_e in 1..E
    return (-lam * s * torch.log(rank.to(torch.float64))).to(torch.float32)


def make_router_inputs(w: Workload, seed: int):
    """x [T, d] (fp32 values, cast later), W_g [d, E] fp32, bias [E] or None (CPU)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(w.T, w.d, generator=g, dtype=torch.float32)
    Wg = torch.randn(w.d, w.E, generator=g, dtype=torch.float32) / math.sqrt(w.d)
    bias = zipf_bias(w.E, w.zipf_s, seed) if w.zipf_s is not None else None
    return x.to(w.torch_act), Wg, bias


def make_expert_weights(w: Workload, seed: int, device="cpu"):
    """W13 [E+S, R, d] and W2 [E+S, d, F] (S shared experts last), drawn expert by expert."""
    if w.expert == "identity":
        return None, None
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed * 1000003 + 1)
    W13 = torch.empty(w.n_experts, w.w13_rows, w.d, dtype=w.torch_act, device=dev)
    W2 = torch.empty(w.n_experts, w.d, w.F, dtype=w.torch_act, device=dev)
    s13, s2 = 1.0 / math.sqrt(w.d), 1.0 / math.sqrt(w.F)
    for e in range(w.n_experts):
        W13[e] = torch.randn(w.w13_rows, w.d, generator=g, device=dev) * s13
        W2[e] = torch.randn(w.d, w.F, generator=g, device=dev) * s2
    return W13, W2


def make_inputs(w: Workload, seed: int = 0, device="cpu") -> dict:
    """All inputs of one workload on ``device``: x, Wg, bias, W13, W2."""
    x, Wg, bias = make_router_inputs(w, seed)
    W13, W2 = make_expert_weights(w, seed, device)
    dev = torch.device(device)
    return dict(
        x=x.to(dev),
        Wg=Wg.to(dev),
        bias=None if bias is None else bias.to(dev),
        W13=W13,
        W2=W2,
    )


def make_stage_inputs(w: Workload, seed: int = 0, device="cpu", rows: int | None = None,
                      keep_frac: float = 0.8) -> dict:
    """Seeded inputs of the stages after the router, drawn directly (no routing):

      topk_idx [T, K] int32: k distinct routed ids per token, drawn with Zipf(s)
                weights over the experts when the workload is skewed, else uniformly;
                the shared slots hold E, E+1, ...
      topk_gate [T, K] fp32: independent draws from U(0.01, 1) (shared slots: 1).
      counts [N] int64: rows per expert for an expert-FFN call, summing to at most
                ``rows`` (default T*K), with some experts left empty.
      xperm [sum(counts), d] act: N(0, 1) rows.
      pos [T*K] int32: a random injective map of a ``keep_frac`` share of the
                assignments onto rows [0, rows); the rest are -1.
      out_rows [rows, d]: N(0, 1) rows in fp32 (cast by the caller to the out dtype).
    """
    g = torch.Generator().manual_seed(1_000_003 + seed)
    T, k, S, E, N = w.T, w.k, w.n_shared, w.E, w.n_experts
    K = k + S
    R = T * K if rows is None else rows
    if w.zipf_s is not None:
        p = torch.arange(1, E + 1, dtype=torch.float64) ** -float(w.zipf_s)
        perm = torch.randperm(E, generator=g)
        weights = torch.empty(E, dtype=torch.float64)
        weights[perm] = p
    else:
        weights = torch.ones(E, dtype=torch.float64)
    idx = torch.multinomial(weights.expand(T, E), k, replacement=False, generator=g).to(torch.int32)
    gate = 0.01 + 0.99 * torch.rand(T, k, generator=g)
    if S:
        idx = torch.cat([idx, (E + torch.arange(S, dtype=torch.int32)).expand(T, S)], dim=1)
        gate = torch.cat([gate, torch.ones(T, S)], dim=1)
    total = int(torch.randint(R // 2, R + 1, (1,), generator=g)) if R > 0 else 0
    empty = torch.rand(N, generator=g) < 0.15
    share = torch.rand(N, generator=g).masked_fill(empty, 0.0)
    if float(share.sum()) == 0.0:
        share[0] = 1.0
    counts = torch.floor(share / share.sum() * total).to(torch.int64)
    A = T * K
    n_keep = min(int(round(keep_frac * A)), R)
    pos = torch.full((A,), -1, dtype=torch.int32)
    chosen = torch.randperm(A, generator=g)[:n_keep]
    pos[chosen] = torch.randperm(R, generator=g)[:n_keep].to(torch.int32)
    dev = torch.device(device)
    return dict(
        topk_idx=idx.contiguous().to(dev),
        topk_gate=gate.to(torch.float32).contiguous().to(dev),
        counts=counts,
        xperm=torch.randn(int(counts.sum()), w.d, generator=g).to(w.torch_act).to(dev),
        pos=pos.to(dev),
        out_rows=torch.randn(R, w.d, generator=g).to(dev),
    )
