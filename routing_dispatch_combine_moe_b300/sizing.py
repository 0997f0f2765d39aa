"""Byte, flop and parameter counts for one MoE layer (host-side arithmetic).

Formulas and where they are stated:

* dispatch bytes per device and direction = T * k * d * bytes_per_element * (D-1)/D
  ("EP Math - Expert Parallelism (MoE)", "The dispatch all-to-all: bytes on the
  wire"); the combine moves the same volume back ("The combine all-to-all: the
  return trip"), so a layer moves twice that.
* per-expert capacity = ceil(f * T * k / E) ("Capacity factor: fixing buffer
  sizes"), optionally floored at a minimum capacity ("MoE Expert Parallelism
  Sizing: Traffic, Capacity, Fabric", "Cross-framework notes").
* gated expert parameters = 3 * d * F ("MoE Expert Parallelism Sizing", "Memory
  residency for the same shape"); the 4d-wide dense FFN expert holds 2 * 4 * d^2
  ("EP Math", "Placing experts across devices").
* expected nodes touched by k uniform picks over n nodes = n (1 - (1 - 1/n)^k), and
  remote nodes = (n - 1)(1 - (1 - 1/n)^k) ("MoE Expert Parallelism Sizing",
  "First-order dispatch and combine bytes").
* imbalance ratio = (max - mean) / mean ("MoE Expert Parallelism Sizing",
  "Rank-level skew and the straggler effect").
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def assignments(T: int, k: int) -> int:
    return T * k


def dispatch_bytes_per_direction(T: int, k: int, d: int, elem_bytes: int, D: int | None = None) -> float:
    """Bytes one device sends in the dispatch all-to-all; D=None counts every assignment."""
    b = T * k * d * elem_bytes
    return b if D is None else b * (D - 1) / D


def layer_comm_bytes(T: int, k: int, d: int, elem_bytes: int, D: int | None = None) -> float:
    """Dispatch plus combine bytes for one layer (two all-to-alls of equal size)."""
    return 2 * dispatch_bytes_per_direction(T, k, d, elem_bytes, D)


def capacity(T: int, k: int, E: int, capacity_factor, min_capacity: int = 0) -> int | None:
    """ceil(f T k / E) with f an exact rational (decimal string, Fraction or int)."""
    if capacity_factor is None:
        return None
    f = Fraction(capacity_factor)
    num, den = f.numerator * T * k, f.denominator * E
    return max(-(-num // den), int(min_capacity))


def capacity_fraction(capacity_factor) -> tuple[int, int]:
    """(numerator, denominator) of the capacity factor, for the C ABI."""
    f = Fraction(capacity_factor)
    return f.numerator, f.denominator


def gated_expert_params(d: int, F: int) -> int:
    return 3 * d * F


def dense4_expert_params(d: int) -> int:
    return 2 * 4 * d * d


def expected_nodes_touched(k: int, n: int) -> float:
    return n * (1 - (1 - 1 / n) ** k)


def expected_remote_nodes(k: int, n: int) -> float:
    return (n - 1) * (1 - (1 - 1 / n) ** k)


def imbalance_ratio(loads) -> float:
    loads = np.asarray(loads, dtype=np.float64)
    mean = loads.mean()
    return float((loads.max() - mean) / mean) if mean > 0 else 0.0


def histogram_summary(counts) -> dict:
    """p50 / p95 / max of a per-expert token histogram, plus its imbalance ratio."""
    c = np.asarray(counts, dtype=np.float64)
    return dict(p50=float(np.percentile(c, 50)), p95=float(np.percentile(c, 95)),
                max=int(c.max()), mean=float(c.mean()), imbalance=imbalance_ratio(c))


# ----------------------------------------------------------- one-GPU algorithmic work
def dispatch_combine_hbm_bytes(T: int, d: int, rows: int, elem_bytes: int) -> int:
    """HBM bytes the on-device dispatch and combine must move at least.

    dispatch reads x (T rows) and writes the dispatched rows; combine reads the
    expert-output rows and writes y (T rows). Routing metadata is not counted.
    """
    return (2 * T + 2 * rows) * d * elem_bytes


def dispatch_hbm_bytes(T: int, d: int, rows: int, elem_bytes: int) -> int:
    return (T + rows) * d * elem_bytes


def combine_hbm_bytes(T: int, d: int, rows: int, elem_bytes: int) -> int:
    return (rows + T) * d * elem_bytes


def expert_gemm_flops(rows: int, d: int, F: int, expert: str) -> tuple[int, int]:
    """(up-projection flops, down-projection flops) over ``rows`` dispatched rows."""
    if expert == "identity":
        return 0, 0
    up_n = 2 * F if expert == "swiglu" else F
    return 2 * rows * d * up_n, 2 * rows * F * d


def router_flops(T: int, d: int, E: int) -> int:
    return 2 * T * d * E


def remote_dispatch_bytes(rank_offsets, d: int, elem_bytes: int, home_rank: int = 0) -> int:
    """Bytes of dispatched rows whose experts live on another virtual rank.

    The device plays ``home_rank`` of D; rank r's rows are
    [rank_offsets[r], rank_offsets[r+1]).
    """
    ro = np.asarray(rank_offsets, dtype=np.int64)
    per_rank = np.diff(ro)
    return int((per_rank.sum() - per_rank[home_rank]) * d * elem_bytes)
