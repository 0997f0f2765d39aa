"""The expert-parallel exchange contract, on CPU with two gloo ranks.

The library lays the dispatched rows out expert-major, so the rows bound for the
owner of experts [r E/D, (r+1) E/D) form one contiguous chunk, starting at
rank_offsets[r]: the "one input chunk per destination" layout an all-to-all takes
("MoE Expert Parallelism Sizing: Traffic, Capacity, Fabric", "First-order dispatch
and combine bytes"; "EP Math - Expert Parallelism (MoE)", "Placing experts across
devices", "The dispatch all-to-all", "The combine all-to-all"). Here each of D = 2
ranks routes its own tokens with the oracle, drops past the capacity before the
exchange, sends each chunk to its owner with all_to_all_single, runs the experts it
owns on what it receives, sends the rows back the same way and combines them. Its y
must equal the single-process oracle forward of the same tokens bit for bit: the
layout and the chunk bookkeeping lose and reorder nothing.

The experts run one row at a time on both sides, so that a BLAS call of another
batch size cannot change a row's rounding.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

D = 2
T, d, E, k, F = 96, 64, 8, 2, 32


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(rank):
    """Shared router and expert weights; each rank's own tokens."""
    g = np.random.default_rng(1234)
    Wg = g.standard_normal((d, E)) / np.sqrt(d)
    W13 = g.standard_normal((E, 2 * F, d)) / np.sqrt(d)
    W2 = g.standard_normal((E, d, F)) / np.sqrt(F)
    x = np.random.default_rng(100 + rank).standard_normal((T, d))
    return x, Wg, W13, W2


def _rowwise_experts(W13, W2):
    from oracle import moe_oracle as orc

    def fn(e, X):
        rows = [orc.expert_swiglu(X[i:i + 1], W13[e, :F].T, W13[e, F:].T, W2[e].T) for i in range(X.shape[0])]
        return np.concatenate(rows, axis=0) if rows else np.zeros((0, d))
    return fn


def _rank_main(rank, port, cf, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(D))
    import torch.distributed as dist
    from oracle import moe_oracle as orc
    dist.init_process_group("gloo")
    try:
        x, Wg, W13, W2 = _inputs(rank)
        fn = _rowwise_experts(W13, W2)
        cap = orc.expert_capacity(T, k, E, cf)
        # route and dispatch locally; drops happen here, before the exchange
        H = orc.router_logits(x, Wg)
        idx = orc.keep_topk(H, k)
        G = orc.kept_softmax(H, idx)
        disp = orc.dispatch(idx, E, cap, D)
        rs = disp["row_src"]
        xperm = x[rs // k]
        ro = disp["rank_offsets"]
        send_rows = [int(ro[r + 1] - ro[r]) for r in range(D)]
        # each destination learns how many rows of each of its experts every sender has
        kept = torch.from_numpy(disp["counts_kept"].astype(np.int64))
        per_expert = torch.empty_like(kept)
        dist.all_to_all_single(per_expert, kept)  # [sender][expert of mine]
        per_expert = per_expert.view(D, E // D).numpy()
        recv_rows = [int(c) for c in per_expert.sum(axis=1)]
        recv = torch.empty(sum(recv_rows), d, dtype=torch.float64)
        dist.all_to_all_single(recv, torch.from_numpy(np.ascontiguousarray(xperm)), recv_rows, send_rows)
        # run the experts this rank owns on each sender's chunk (expert-major inside it)
        out_recv = torch.empty_like(recv)
        at = 0
        for s in range(D):
            for j in range(E // D):
                n = int(per_expert[s, j])
                e = rank * (E // D) + j
                out_recv[at:at + n] = torch.from_numpy(fn(e, recv[at:at + n].numpy()))
                at += n
        # send the outputs back; each comes back to the row it left from
        out = torch.empty(xperm.shape[0], d, dtype=torch.float64)
        dist.all_to_all_single(out, out_recv, send_rows, recv_rows)
        y = orc.combine(G, disp["pos"], out.numpy(), T, k)
        ref = orc.moe_forward(x, Wg, k, fn, capacity=cap, D=D)
        q.put((rank, bool(np.array_equal(y, ref["y"])), int(disp["n_dropped"]), send_rows, recv_rows,
               float(np.abs(y - ref["y"]).max())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("cf", [None, "1"])
def test_two_ranks_exchange_rank_chunks_and_match_the_single_process_forward(cf):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, cf, q)) for r in range(D)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, equal, dropped, send_rows, recv_rows, err in res:
        assert equal, f"rank {rank}: y differs from the single-process forward by {err:.3e}"
        assert sum(send_rows) == T * k - dropped
        if cf is not None:
            assert dropped > 0  # capacity factor 1 drops some of each rank's assignments
    # what one rank sends to the other is what the other receives from it
    assert res[0][3][1] == res[1][4][0] and res[1][3][0] == res[0][4][1]


# ----------------------------------------------------------------- deduplicated dispatch
K_DD = 4  # four slots per token, so a token often uses several experts of one rank


def _dedup_rank_main(rank, port, q):
    """Deduplicated exchange: token t sends its row once to each rank that holds one of
    its kept routed experts ("MoE Expert Parallelism Sizing: Traffic, Capacity, Fabric",
    "First-order dispatch and combine bytes": the dispatch carries one copy per
    destination), with the token's expert ids beside it; the receiver fans the row out to
    each of its own experts the token uses, and returns one output row per assignment
    (the combine is not deduplicated)."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(D))
    import torch.distributed as dist
    from oracle import moe_oracle as orc
    dist.init_process_group("gloo")
    try:
        x, Wg, W13, W2 = _inputs(rank)
        fn = _rowwise_experts(W13, W2)
        cap = orc.expert_capacity(T, K_DD, E, "1")
        H = orc.router_logits(x, Wg)
        idx = orc.keep_topk(H, K_DD)
        G = orc.kept_softmax(H, idx)
        disp = orc.dispatch(idx, E, cap, D)
        pos = disp["pos"]
        dd = orc.dedup_send(idx, pos, E, D)
        per_rank = E // D
        send_src = np.asarray(dd["send_src"], np.int64)
        tok = send_src // D
        dest = send_src % D
        send_counts = [int(c) for c in dd["send_counts"]]
        # each send row carries its token's kept expert ids on the destination (-1 elsewhere)
        kept = (pos.reshape(T, K_DD) >= 0)
        meta = np.where(kept[tok] & (idx[tok] // per_rank == dest[:, None]), idx[tok], -1)
        counts = torch.tensor(send_counts, dtype=torch.int64)
        recv_counts_t = torch.empty_like(counts)
        dist.all_to_all_single(recv_counts_t, counts)
        recv_counts = [int(c) for c in recv_counts_t]
        rows = torch.empty(sum(recv_counts), d, dtype=torch.float64)
        dist.all_to_all_single(rows, torch.from_numpy(np.ascontiguousarray(x[tok])), recv_counts, send_counts)
        rmeta = torch.empty(sum(recv_counts), K_DD, dtype=torch.int64)
        dist.all_to_all_single(rmeta, torch.from_numpy(np.ascontiguousarray(meta)), recv_counts, send_counts)
        rows, rmeta = rows.numpy(), rmeta.numpy()
        # fan out: one output per (received row, local slot), in received order, slots ascending
        back = [fn(int(e), rows[i:i + 1])[0] for i in range(rows.shape[0]) for e in rmeta[i] if e >= 0]
        back_counts = []
        at = 0
        for s in range(D):
            seg = rmeta[at:at + recv_counts[s]]
            back_counts.append(int((seg >= 0).sum()))
            at += recv_counts[s]
        ret_counts = [int((meta[dest == r] >= 0).sum()) for r in range(D)]
        ret = torch.empty(sum(ret_counts), d, dtype=torch.float64)
        send_back = torch.from_numpy(np.asarray(back, np.float64).reshape(-1, d))
        dist.all_to_all_single(ret, send_back, ret_counts, back_counts)
        # the returned rows follow this rank's send rows (rank-major) and their slots in order
        out = np.zeros((int(pos.max()) + 1 if (pos >= 0).any() else 0, d))
        at = 0
        for i in range(send_src.size):
            for j in range(K_DD):
                if meta[i, j] >= 0:
                    out[pos[tok[i] * K_DD + j]] = ret[at].numpy()
                    at += 1
        y = orc.combine(G, pos, out, T, K_DD)
        ref = orc.moe_forward(x, Wg, K_DD, fn, capacity=cap, D=D)
        n_kept = int((pos >= 0).sum())
        q.put((rank, bool(np.array_equal(y, ref["y"])), int(dd["n_send"]), n_kept, send_counts, recv_counts,
               float(np.abs(y - ref["y"]).max())))
    finally:
        dist.destroy_process_group()


def test_two_ranks_deduplicated_exchange_matches_the_single_process_forward():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dedup_rank_main, args=(r, port, q)) for r in range(D)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, equal, n_send, n_kept, send_counts, recv_counts, err in res:
        assert equal, f"rank {rank}: y differs from the single-process forward by {err:.3e}"
        assert sum(send_counts) == n_send
        # at most one row per (token, rank): fewer rows than kept assignments travel
        assert n_send <= T * D and n_send < n_kept
    assert res[0][4][1] == res[1][5][0] and res[1][4][0] == res[0][5][1]
