"""CPU oracle for the forward pass of one top-k-routed Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE. This module is a plain, slow, float64 statement of what the
layer computes, used only to check the CUDA library. Only the test suite, the
package's ``smoke()`` entry and ``bench.py``'s CPU-baseline leg may import it; the
library itself never does, and it shares no code, table or helper with the CUDA
path. It does not import the library or its input generator: every function takes
plain arrays.

Sources (page title, then section):

* [GATE]  "Mixture-of-Experts (MoE) Architecture and Expert Parallelism",
          section 2 "The Gating Network Formulation": H(x) = x W_g + eps,
          G(x) = Softmax(KeepTopK(H(x), K)), y = sum_{i in TopK} G_i(x) Expert_i(x);
          KeepTopK keeps the K largest coordinates and sets the rest to -inf.
* [EPSH]  "EP Math - Expert Parallelism (MoE)", "What expert parallelism actually
          shards" and "Placing experts across devices": E experts, each a complete FFN,
          E/D whole experts per device, E divisible by D.
* [CAP]   same page, "Capacity factor: fixing buffer sizes": C = f * N * k / E,
          rounded up.
* [DROP]  same page, "Token drop: what overflow costs": an assignment past the
          capacity is skipped by its expert and adds nothing to y, the same as a
          zero expert output (the token still passes through the residual, which
          the caller adds).
* [A2A]   same page, "The dispatch all-to-all" / "The combine all-to-all": each
          assignment is a d-vector sent to its expert; the combine weights the k
          returned vectors by the gates and sums them.
* [MINC]  "MoE Expert Parallelism Sizing: Traffic, Capacity, Fabric",
          "Cross-framework notes": a minimum capacity per expert regardless of the
          capacity factor.
* [SWI]   same page, "Memory residency for the same shape": the gated three-matrix
          expert form (gate, up, down).
* [SHR]   same page, "Token assignments and the capacity worksheet" and "Training,
          prefill and decode are different workloads": a shared expert that every
          token uses; in DeepSeek's decode deployment it is handled like a routed
          one, so each token sends 9 vectors (8 routed + the shared expert).
* [NODE]  same page, "First-order dispatch and combine bytes" (the node-limited
          rows): each token is dispatched to at most M nodes (DeepSeek-V3: 4);
          Megatron calls the same constraint group-limited routing.
* [DEDUP] same page, same section (the deduplicated rows): a token goes once to
          each destination node that holds any of its experts, so 8 uniformly
          random experts over 8 nodes touch 8 (1 - (7/8)^8) ~ 5.25 nodes, of which
          7 (1 - (7/8)^8) ~ 4.6 are remote.
* [FP8]   same page, same section and "Decode": FP8 dispatch sends the token rows in
          FP8 (e4m3) with scale tensors, halving the dispatch bytes, while the
          combine may stay in BF16; the decode example counts 128-element blocks.

Readings where the pages are silent (each is listed in the design notes too):

* ties in KeepTopK go to the lower expert id, and the kept slots are ordered by
  descending logit;
* the optional per-expert router bias is added to H before KeepTopK, so it enters
  both the selection and the softmax, like the eps term;
* overflow is dropped in ascending token order: an expert keeps its first C
  assignments by token index;
* rows are ordered by (expert, token); the list of dropped assignments is ordered
  the same way (expert, then token);
* a dropped slot's gate is not renormalised over the kept slots;
* SwiGLU expert: silu(x W_gate) * (x W_up) then W_down, silu(z) = z / (1 + e^-z),
  no biases; ReLU expert: relu(x W_1) W_2.
* shared experts are experts E .. E+n_shared-1: every token is also dispatched to
  each of them with gate 1, after its k routed slots; capacity limits only the
  routed experts.
* drop by gate [SIZ "Capacity semantics decide what crosses the wire": overflow
  dropped by selected probability]: an overflowing expert keeps the C assignments
  with the largest gates, equal gates going to the lower token index; its kept rows
  stay in token order;
* padded layout [CAP: every expert's buffer holds C token slots, under-full experts
  padded]: expert e's kept rows start at row e*C, the rest of its C rows are zero.
* group-limited routing [NODE] (the pages name the constraint, not the rule): the
  E experts form G equal contiguous groups; a group's score is its largest logit;
  a token keeps the M groups with the largest scores (equal scores: lower group
  first) and KeepTopK runs over the experts of those groups only. This is the same
  as walking the experts in KeepTopK order and skipping an expert whose group would
  be the (M+1)-th distinct group. The gates are the kept softmax over the k kept
  logits, as without the limit.
* FP8 dispatch [FP8] (the pages give the format, not the scale rule): every
  128-element block of a token row (the last block of a row may be shorter) gets
  a power-of-two scale 2^s, s the smallest integer with amax / 2^s <= 448 (448 is
  e4m3's largest finite value; an all-zero block takes s = 0); each element is
  x / 2^s rounded to the nearest e4m3 value (ties to the even code); the receiver
  multiplies back by 2^s, which is exact, so the experts see q * 2^s.
* FP8 expert GEMM ([FP8], and "Memory residency for the same shape" of the same page,
  which sizes the experts' weights in FP8 with scale tensors; the scale granularity
  of the GEMM's operands is ours): the same rule with one block per row. Every dispatched
  row (routed and shared) is q * 2^s with one s per token row, and the up projection's
  weights are quantized per output channel (one s per row of W13) the same way; the
  up projection then multiplies those exact values, h and the down projection are
  as in the bf16 path.
* FP8 down projection (the same pages; ours too): h, as the bf16 value the up
  projection stores, is quantized per row by the same rule, and W2 per output channel
  (one s per row of W2 [d, F]); the down projection multiplies those values. The bf16
  rounding comes first because h is stored in bf16 before it is quantized: the
  e4m3 decision is taken on the stored value (``fp8_hidden``).
* deduplicated dispatch [DEDUP]: with D virtual ranks (rank r owns routed experts
  [r E/D, (r+1) E/D)), token t sends one row to rank r when at least one of its
  kept routed assignments lives there; send rows are rank-major, in token order
  inside a rank's chunk; the receiving rank copies that row to each of the token's
  expert rows it holds. Shared experts are replicated, so they take their rows from
  x directly and send nothing.

Every arithmetic step runs in float64 on exact float64 copies of the inputs (bf16
and fp32 values are exact in float64). ``round_to_bf16`` is only for the optional
"faithful" diagnostic that rounds at the points where the GPU rounds.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

__all__ = [
    "router_logits",
    "keep_topk",
    "kept_softmax",
    "expert_capacity",
    "dispatch",
    "expert_relu",
    "expert_swiglu",
    "silu",
    "combine",
    "moe_forward",
    "near_tie_flags",
    "keep_topk_grouped",
    "group_allowed",
    "group_tie_flags",
    "dedup_send",
    "e4m3_values",
    "quantize_fp8_blocks",
    "quantize_fp8_rows",
    "fp8_hidden",
    "round_to_bf16",
]


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------- router
def router_logits(x, Wg, bias=None) -> np.ndarray:
    """H = x . W_g (+ b), [T, E] float64.  [GATE]: H(x) = x W_g + eps with eps = 0.

    ``x`` is [T, d], ``Wg`` is [d, E] (the page's W_g in R^{d x E}); ``bias`` is an
    optional [E] per-expert term added to every token's logits.
    """
    H = _f64(x) @ _f64(Wg)
    if bias is not None:
        H = H + _f64(bias)[None, :]
    return H


def keep_topk(H, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, [T, k] int64.  [GATE] KeepTopK.

    Slot j holds the (j+1)-th largest logit. Equal logits rank the lower expert id
    first: the sort key is (-H[t, e], e), ascending.
    """
    H = _f64(H)
    T, E = H.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    expert_id = np.broadcast_to(np.arange(E), H.shape)
    order = np.lexsort((expert_id, -H), axis=-1)  # last key is the primary key
    return order[:, :k].astype(np.int64)


def kept_softmax(H, idx) -> np.ndarray:
    """Gates G = Softmax(KeepTopK(H)), returned at the kept slots, [T, k].  [GATE]

    Written as the definition: every coordinate outside the top k is set to -inf,
    a softmax runs over all E coordinates (exp(-inf) = 0), and the kept entries are
    read back in slot order.
    """
    H = _f64(H)
    T, E = H.shape
    rows = np.arange(T)[:, None]
    masked = np.full_like(H, -np.inf)
    masked[rows, idx] = H[rows, idx]
    shifted = masked - masked.max(axis=1, keepdims=True)
    p = np.exp(shifted)
    G = p / p.sum(axis=1, keepdims=True)
    return G[rows, idx]


def near_tie_flags(H, k: int, rel: float = 1e-6):
    """Tokens whose top-k selection or slot order rests on a near tie.

    Returns (set_tie, order_tie), both [T] bool. ``set_tie``: the k-th and (k+1)-th
    largest logits differ by less than ``rel`` relative to the larger magnitude, so
    a different but equally valid rounding could pick another set. ``order_tie``:
    two adjacent kept logits are that close, so the slot order could differ.
    """
    H = _f64(H)
    T, E = H.shape
    s = -np.sort(-H, axis=1)

    def close(a, b):
        scale = np.maximum(np.abs(a), np.abs(b))
        return (a - b) < rel * scale

    set_tie = np.zeros(T, bool) if k >= E else close(s[:, k - 1], s[:, k])
    order_tie = np.zeros(T, bool)
    for j in range(k - 1):
        order_tie |= close(s[:, j], s[:, j + 1])
    return set_tie, order_tie


def keep_topk_grouped(H, k: int, n_groups: int, topk_groups: int) -> np.ndarray:
    """Group-limited KeepTopK, [T, k] int64.  [NODE]

    The experts form ``n_groups`` contiguous groups of E / n_groups. Each group is
    scored by its largest logit; the ``topk_groups`` best groups are kept (equal
    scores: lower group first), every logit outside them is set to -inf, and
    KeepTopK runs on what is left.
    """
    H = _f64(H)
    T, E = H.shape
    if n_groups < 1 or E % n_groups:
        raise ValueError("the groups must split the experts evenly")
    gs = E // n_groups
    if not 1 <= topk_groups <= n_groups or k > topk_groups * gs:
        raise ValueError("need 1 <= topk_groups <= n_groups and k <= topk_groups * E / n_groups")
    return keep_topk(np.where(group_allowed(H, n_groups, topk_groups), H, -np.inf), k)


def group_allowed(H, n_groups: int, topk_groups: int) -> np.ndarray:
    """[T, E] bool: the experts of each token's ``topk_groups`` best groups.  [NODE]"""
    H = _f64(H)
    T, E = H.shape
    gs = E // n_groups
    score = H.reshape(T, n_groups, gs).max(axis=2)
    order = np.argsort(-score, axis=1, kind="stable")  # stable: equal scores keep the lower group first
    kept_group = np.zeros((T, n_groups), bool)
    np.put_along_axis(kept_group, order[:, :topk_groups], True, axis=1)
    return np.repeat(kept_group, gs, axis=1)


def group_tie_flags(H, n_groups: int, topk_groups: int, rel: float = 1e-6) -> np.ndarray:
    """Tokens whose group choice rests on a near tie: the topk_groups-th and the next
    group score differ by less than ``rel`` relative to the larger magnitude. [T] bool."""
    H = _f64(H)
    T, E = H.shape
    if topk_groups >= n_groups:
        return np.zeros(T, bool)
    score = -np.sort(-H.reshape(T, n_groups, E // n_groups).max(axis=2), axis=1)
    a, b = score[:, topk_groups - 1], score[:, topk_groups]
    return (a - b) < rel * np.maximum(np.abs(a), np.abs(b))


# ------------------------------------------------------------------------- dispatch
def expert_capacity(T: int, k: int, E: int, capacity_factor, min_capacity: int = 0):
    """Per-expert capacity C = ceil(f * T * k / E), floored at ``min_capacity``.

    [CAP] gives C = f N k / E rounded up (N = the tokens this device holds here);
    [MINC] adds the floor. ``capacity_factor`` None means dropless (returns None).
    The factor is taken as an exact rational: a decimal string such as "1.25", a
    Fraction, or an int; a float is converted by its exact binary value.
    """
    if capacity_factor is None:
        return None
    f = Fraction(capacity_factor)
    if f < 0:
        raise ValueError("capacity factor must be >= 0")
    C = math.ceil(f * T * k / E)
    return max(C, int(min_capacity))


def dispatch(idx, E: int, capacity=None, D: int = 1, capped_experts=None, gates=None,
             drop_policy: str = "token", layout: str = "packed") -> dict:
    """Group the T*k assignments by expert, dropping overflow.  [A2A], [CAP], [DROP]

    Assignment a = t*k + j is token t's j-th slot. For each expert in ascending id
    the assignments routed to it are listed by ascending token index; the first
    ``capacity`` of them are kept (all of them when ``capacity`` is None) and the
    rest are dropped. Kept assignments take consecutive rows in that order, so the
    row segment of expert e is [offsets[e], offsets[e+1]). With D virtual ranks,
    rank r owns experts [r E/D, (r+1) E/D) [EPSH], and its rows start at
    rank_offsets[r]. Only experts with id < ``capped_experts`` (default: all E) are
    held to the capacity; the ranks then split those experts, and later experts
    (shared ones) follow after rank_offsets[D].

    ``drop_policy`` "gate" keeps, per overflowing expert, the ``capacity``
    assignments with the largest ``gates`` (equal gates: lower token first) instead
    of the first ones by token; kept rows stay in token order. ``layout`` "padded"
    gives every expert a fixed segment of ``capacity`` rows starting at e*C (offsets
    are e*C); rows past an expert's kept count are padding.
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    capped = E if capped_experts is None else capped_experts
    if capped % D != 0:
        raise ValueError("the routed experts must divide into D ranks")
    if layout == "padded" and (capacity is None or capped != E):
        raise ValueError("the padded layout needs a capacity and no uncapped experts")
    if drop_policy == "gate":
        gates = np.asarray(gates, np.float64).reshape(T, k)
    counts_routed = np.zeros(E, np.int64)
    counts_kept = np.zeros(E, np.int64)
    kept_ids, dropped_ids = [], []
    for e in range(E):
        tok, slot = np.nonzero(idx == e)  # row-major scan: ascending token index
        a = tok * k + slot
        counts_routed[e] = a.size
        if capacity is None or e >= capped or a.size <= capacity:
            keep, drop = a, a[:0]
        elif drop_policy == "token":
            keep, drop = a[:capacity], a[capacity:]
        else:
            by_gate = np.lexsort((tok, -gates[tok, slot]))  # primary: gate desc; then token asc
            chosen = np.zeros(a.size, bool)
            chosen[by_gate[:capacity]] = True
            keep, drop = a[chosen], a[~chosen]  # both still in token order
        counts_kept[e] = keep.size
        kept_ids.append(keep)
        dropped_ids.append(drop)
    drop_list = np.concatenate(dropped_ids).astype(np.int64)
    pos = np.full(T * k, -1, np.int64)
    if layout == "padded":
        offsets = np.arange(E + 1, dtype=np.int64) * capacity
        row_src = np.full(E * capacity, -1, np.int64)
        for e in range(E):
            row_src[offsets[e]:offsets[e] + kept_ids[e].size] = kept_ids[e]
        valid = row_src >= 0
        pos[row_src[valid]] = np.nonzero(valid)[0]
    else:
        row_src = np.concatenate(kept_ids).astype(np.int64)
        offsets = np.concatenate([[0], np.cumsum(counts_kept)]).astype(np.int64)
        pos[row_src] = np.arange(row_src.size)
    rank_offsets = offsets[np.arange(D + 1) * (capped // D)]
    return dict(
        counts_routed=counts_routed,
        counts_kept=counts_kept,
        offsets=offsets,
        row_src=row_src,
        pos=pos,
        drop_list=drop_list,
        n_dropped=int(drop_list.size),
        rank_offsets=rank_offsets,
        capacity=capacity,
        layout=layout,
    )


def dedup_send(idx, pos, n_routed: int, D: int) -> dict:
    """Deduplicated dispatch: one row per (token, destination rank).  [DEDUP]

    ``idx`` [T, K] and ``pos`` [T*K] come from KeepTopK and ``dispatch``; experts
    below ``n_routed`` are routed and split over D ranks, E/D each (rank r holds
    [r n_routed/D, (r+1) n_routed/D)); higher ids are shared experts, which send
    nothing. Token t sends its row to rank r when one of its kept routed assignments
    lives there. Returns:
      sent          [T, D] bool
      send_counts   [D] rows sent to each rank
      send_offsets  [D+1] exclusive scan of send_counts
      send_pos      [T*D] send row of (t, r), -1 when t sends nothing to r
      send_src      [n_send] t*D + r of each send row (rank-major, then token)
      fan_src       [T*K] send row feeding each kept routed assignment, else -1
      n_send
    """
    idx = np.asarray(idx, np.int64)
    T, K = idx.shape
    pos = np.asarray(pos, np.int64).reshape(T, K)
    if n_routed % D:
        raise ValueError("the routed experts must divide into D ranks")
    per_rank = n_routed // D
    sent = np.zeros((T, D), bool)
    for t in range(T):
        for j in range(K):
            if pos[t, j] >= 0 and idx[t, j] < n_routed:
                sent[t, idx[t, j] // per_rank] = True
    send_counts = sent.sum(axis=0).astype(np.int64)
    send_offsets = np.concatenate([[0], np.cumsum(send_counts)]).astype(np.int64)
    send_pos = np.full(T * D, -1, np.int64)
    send_src = []
    for r in range(D):
        for t in range(T):
            if sent[t, r]:
                send_pos[t * D + r] = len(send_src)
                send_src.append(t * D + r)
    fan_src = np.full(T * K, -1, np.int64)
    for t in range(T):
        for j in range(K):
            if pos[t, j] >= 0 and idx[t, j] < n_routed:
                fan_src[t * K + j] = send_pos[t * D + idx[t, j] // per_rank]
    return dict(sent=sent, send_counts=send_counts, send_offsets=send_offsets, send_pos=send_pos,
                send_src=np.asarray(send_src, np.int64), fan_src=fan_src, n_send=len(send_src))


# ------------------------------------------------------------------- FP8 dispatch
def e4m3_values() -> np.ndarray:
    """The value of each of the 256 e4m3 codes (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits; exponent 0 is subnormal, m * 2^-9; codes 0x7F and 0xFF are NaN,
    there is no infinity), float64.  [FP8]"""
    v = np.empty(256)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        ex, man = (c >> 3) & 0xF, c & 0x7
        if ex == 0xF and man == 0x7:
            v[c] = np.nan
        elif ex == 0:
            v[c] = sign * man * 2.0 ** -9
        else:
            v[c] = sign * (1 + man / 8) * 2.0 ** (ex - 7)
    return v


def _e4m3_round(a) -> np.ndarray:
    """Code of the nearest finite e4m3 value to each element: the magnitude is rounded
    to the nearest of the codes 0x00..0x7E (ties: the even code), then the sign bit is
    set for negative inputs (-0.0 included), as an IEEE-style rounding does.

    Code c (0 <= c < 0x7E) is nearest for the magnitudes from the midpoint between
    codes c - 1 and c to the midpoint between c and c + 1; a magnitude exactly on a
    midpoint goes to the even code of the two; magnitudes at or past the midpoint
    below 448 go to 448 (0x7E), the largest finite value."""
    a = np.asarray(a, np.float64)
    mags = e4m3_values()[:0x7F]           # codes 0x00..0x7E, increasing magnitudes
    mid = (mags[:-1] + mags[1:]) / 2.0    # mid[c] lies between codes c and c + 1
    m = np.abs(a).ravel()
    pick = np.searchsorted(mid, m, side="left")        # the first code whose upper midpoint is >= m
    on_mid = (pick < mid.size) & (m == mid[np.minimum(pick, mid.size - 1)])
    pick = pick + (on_mid & (pick % 2 == 1))           # a tie between codes pick and pick + 1: the even one
    neg = np.signbit(a.ravel())
    return (pick | np.where(neg, 0x80, 0)).astype(np.uint8).reshape(a.shape)


def quantize_fp8_blocks(x, block: int = 128) -> dict:
    """Per-block e4m3 quantization of the rows of ``x`` [rows, d].  [FP8]

    Returns codes [rows, d] uint8, scale exponents s [rows, ceil(d/block)] int64, the
    scales 2^s (float64) and the dequantized rows q * 2^s (float64).
    """
    x = _f64(x)
    rows, d = x.shape
    nb = -(-d // block)
    # every block of every row at once: the row padded with zeros to nb whole blocks (a
    # zero changes no block's amax; the padding's codes are dropped)
    xb = np.zeros((rows, nb * block))
    xb[:, :d] = x
    xb = xb.reshape(rows, nb, block)
    amax = np.abs(xb).max(axis=2)
    nz = amax > 0
    s = np.zeros((rows, nb), np.int64)
    s[nz] = np.ceil(np.log2(amax[nz] / 448.0)).astype(np.int64)
    while True:  # guard the log against rounding: the smallest s with amax / 2^s <= 448
        up = nz & (np.ldexp(amax, -s) > 448.0)
        down = nz & (np.ldexp(amax, -(s - 1)) <= 448.0)
        if not (up.any() or down.any()):
            break
        s = s + up - down
    codes = _e4m3_round(np.ldexp(xb, -s[:, :, None])).reshape(rows, nb * block)[:, :d]
    vals = e4m3_values()
    deq = np.ldexp(vals[codes].reshape(rows, -1), np.repeat(s, block, axis=1)[:, :d])
    return dict(codes=np.ascontiguousarray(codes), exps=s, scales=np.ldexp(1.0, s), deq=deq)


def quantize_fp8_rows(x, chunk: int = 2048) -> dict:
    """Row-wise e4m3 quantization: the [FP8] rule of quantize_fp8_blocks with one block
    per row (one scale 2^s per row). Rows are independent; they are taken ``chunk`` at a
    time only to bound the memory of the float64 temporaries.

    Returns codes [rows, d] uint8, exponents s [rows] int64, scales 2^s and the
    dequantized rows q * 2^s (float64).
    """
    x = _f64(x)
    rows, d = x.shape
    exps = np.zeros(rows, np.int64)
    codes = np.zeros((rows, d), np.uint8)
    vals = e4m3_values()
    for r0 in range(0, rows, chunk):
        seg = x[r0:r0 + chunk]
        amax = np.abs(seg).max(axis=1) if d else np.zeros(seg.shape[0])
        nz = amax > 0
        s = np.zeros(seg.shape[0], np.int64)
        s[nz] = np.ceil(np.log2(amax[nz] / 448.0)).astype(np.int64)
        while True:  # guard the log against rounding: the smallest s with amax / 2^s <= 448
            up = nz & (np.ldexp(amax, -s) > 448.0)
            down = nz & (np.ldexp(amax, -(s - 1)) <= 448.0)
            if not (up.any() or down.any()):
                break
            s = s + up - down
        exps[r0:r0 + chunk] = s
        codes[r0:r0 + chunk] = _e4m3_round(np.ldexp(seg, -s[:, None]))
    deq = np.ldexp(vals[codes], exps[:, None])
    return dict(codes=codes, exps=exps, scales=np.ldexp(1.0, exps), deq=deq)


def fp8_hidden(h) -> np.ndarray:
    """The FP8 form of the hidden activation: each row of h rounded to bf16 (where the up
    projection stores it), then quantized per row (``quantize_fp8_rows``); float64."""
    return quantize_fp8_rows(round_to_bf16(h))["deq"]


# -------------------------------------------------------------------------- experts
def silu(z):
    """silu(z) = z / (1 + e^-z)."""
    z = _f64(z)
    return z / (1.0 + np.exp(-z))


def hidden_relu(X, W1) -> np.ndarray:
    """Hidden activation of the ReLU expert: h = relu(X W1), W1 [d, F]."""
    return np.maximum(_f64(X) @ _f64(W1), 0.0)


def hidden_swiglu(X, Wgate, Wup) -> np.ndarray:
    """Hidden activation of the gated expert [SWI]: h = silu(X Wgate) * (X Wup)."""
    X = _f64(X)
    return silu(X @ _f64(Wgate)) * (X @ _f64(Wup))


def expert_relu(X, W1, W2, hidden=None) -> np.ndarray:
    """ReLU FFN expert: relu(X W1) W2, with W1 [d, F] and W2 [F, d]. ``hidden``, if
    given, maps h before the down projection (``fp8_hidden`` for the FP8 down projection)."""
    h = hidden_relu(X, W1)
    if hidden is not None:
        h = hidden(h)
    return h @ _f64(W2)


def expert_swiglu(X, Wgate, Wup, Wdown, faithful: bool = False, hidden=None) -> np.ndarray:
    """Gated expert [SWI]: (silu(X Wgate) * (X Wup)) Wdown; Wgate, Wup [d, F], Wdown [F, d].

    ``faithful`` rounds the hidden activation to bf16 before the down projection,
    where the GPU path stores it (diagnostic only). ``hidden``, if given, maps h before
    the down projection (``fp8_hidden`` for the FP8 down projection).
    """
    h = hidden_swiglu(X, Wgate, Wup)
    if faithful:
        h = round_to_bf16(h)
    if hidden is not None:
        h = hidden(h)
    return h @ _f64(Wdown)


# -------------------------------------------------------------------------- combine
def combine(G, pos, out, T: int, k: int) -> np.ndarray:
    """y_t = sum over kept slots j of G[t, j] * out[pos[t, j]].  [GATE], [A2A], [DROP]

    A dropped slot (pos = -1) contributes nothing and the remaining gates are not
    renormalised. Slots are added in slot order.
    """
    out = _f64(out)
    G = _f64(G)
    pos = np.asarray(pos).reshape(T, k)
    y = np.zeros((T, out.shape[1]), np.float64)
    for j in range(k):
        p = pos[:, j]
        kept = p >= 0
        y[kept] += G[kept, j, None] * out[p[kept]]
    return y


def moe_forward(x, Wg, k: int, expert_fn, capacity=None, bias=None, D: int = 1, n_shared: int = 0,
                drop_policy: str = "token", layout: str = "packed", n_groups: int = 0,
                topk_groups: int = 0, dispatch_dtype: str = "act") -> dict:
    """The whole layer: logits, KeepTopK, kept softmax, dispatch, experts, combine.

    ``expert_fn(e, X)`` returns Expert_e applied to the rows X (an [M, d] float64
    array); for identity experts pass ``lambda e, X: X``. With ``n_shared`` shared
    experts [SHR], every token also uses experts E .. E+n_shared-1 with gate 1 in
    slots k .. k+n_shared-1. With ``topk_groups`` (0 < topk_groups < n_groups) the
    selection is group-limited [NODE]. Returns every intermediate the GPU path
    exposes, in float64 (y is not rounded); ``idx`` and ``G`` then have k + n_shared
    slots. The deduplicated send buffer changes where rows travel, not their values,
    so y does not depend on it (``dedup_send`` describes it). With ``dispatch_dtype``
    "fp8" the rows travel as per-block e4m3 codes [FP8] and the experts receive the
    dequantized rows; shared experts are replicated and read x itself. With
    "fp8_gemm" every kept row (shared ones too) is the row-quantized token row
    (``quantize_fp8_rows``); ``expert_fn`` then stands for the FP8 experts (their up
    weights quantized per output channel, see packed.expert_fn).
    """
    x = _f64(x)
    T, d = x.shape
    H = router_logits(x, Wg, bias)
    E = H.shape[1]
    if n_groups and 0 < topk_groups < n_groups:
        idx = keep_topk_grouped(H, k, n_groups, topk_groups)
    else:
        idx = keep_topk(H, k)
    G = kept_softmax(H, idx)
    if n_shared:
        idx = np.concatenate([idx, np.broadcast_to(E + np.arange(n_shared), (T, n_shared))], axis=1)
        G = np.concatenate([G, np.ones((T, n_shared))], axis=1)
        k = k + n_shared
    disp = dispatch(idx, E + n_shared, capacity, D, capped_experts=E, gates=G, drop_policy=drop_policy,
                    layout=layout)
    rs = disp["row_src"]
    xperm = np.zeros((rs.size, d))
    xperm[rs >= 0] = x[rs[rs >= 0] // k]  # padding rows (row_src -1) stay zero
    if dispatch_dtype == "fp8":
        xq = quantize_fp8_blocks(x)["deq"]
        routed = (rs >= 0) & (idx.reshape(-1)[np.maximum(rs, 0)] < E)
        xperm[routed] = xq[rs[routed] // k]
    elif dispatch_dtype == "fp8_gemm":
        xq = quantize_fp8_rows(x)["deq"]
        xperm[rs >= 0] = xq[rs[rs >= 0] // k]
    out = np.zeros_like(xperm)
    off = disp["offsets"]
    for e in range(E + n_shared):
        lo, hi = off[e], off[e + 1]
        if hi > lo:
            out[lo:hi] = expert_fn(e, xperm[lo:hi])
    y = combine(G, disp["pos"], out, T, k)
    res = dict(H=H, idx=idx, G=G, xperm=xperm, out=out, y=y)
    res.update(disp)
    return res


# ----------------------------------------------------------------------- diagnostics
def round_to_bf16(a) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned as float64.

    Goes through float32 first (as the GPU does: its values are fp32 before the
    store). Used only by the faithful diagnostic and by tests that state a
    result in the bf16 output format.
    """
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    out = r.view(np.float32).astype(np.float64)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = np.nan
    return out
