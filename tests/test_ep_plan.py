"""Expert parallelism, host side (no GPU): the library's plan of every pair's row
at its owner (mm_moe_ep_plan) against the oracle's routing of all ranks' tokens
together, in one process for 1, 2 and 4 ranks and across two gloo processes that
exchange their counts and metadata as a multi-GPU run would."""
import os
import socket

import numpy as np
import pytest
import torch

import oracle as O


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


def _routing(seed, T, K, E, masked=0.1):
    g = np.random.default_rng(seed)
    idx = np.stack([g.permutation(E)[:K] for _ in range(T)]).astype(np.int32) if T else np.zeros((0, K), np.int32)
    if T:
        idx[g.random((T, K)) < masked] = -1
    w = g.random((T, K)).astype(np.float32)
    return idx, w


def _expected(idx_all, T, K, E, N):
    """From the oracle's routing of every rank's tokens (rank-major), unpadded
    (block 1): each pair's row at its owner and each owner's rows."""
    r = O.route(idx_all, E, 1)
    Eloc = E // N
    first = r["blk_off"][np.arange(N) * Eloc]            # first global row of each owner's experts
    owner = np.where(idx_all >= 0, idx_all // Eloc, -1)
    send = np.where(r["slot"] >= 0, r["slot"] - first[np.maximum(owner, 0)], -1)
    rows = [int(r["blk_off"][(o + 1) * Eloc] - first[o]) for o in range(N)]
    return r, first, send, rows


@pytest.mark.parametrize("N", [1, 2, 4])
def test_plan_matches_oracle_routing(M, N):
    T, K, E = 37, 3, 8
    per_rank = [_routing(100 + r, T, K, E) for r in range(N)]
    idx_all = np.concatenate([p[0] for p in per_rank])
    counts_all = np.stack([np.bincount(p[0][p[0] >= 0], minlength=E) for p in per_rank]).astype(np.int32)
    r, first, send, rows = _expected(idx_all, T, K, E, N)
    Eloc = E // N
    for rank in range(N):
        send_row, nrows, rex = M.mm_moe_ep_plan(counts_all, per_rank[rank][0], T, K, E, N, rank)
        assert np.array_equal(send_row, send[rank * T:(rank + 1) * T].reshape(-1))
        assert nrows == rows[rank]
        # every received row's expert, from the oracle's pool order
        gl = first[rank] + np.arange(nrows)
        src = r["src"][gl]
        assert np.all(src >= 0)
        assert np.array_equal(rex, idx_all.reshape(-1)[src] - rank * Eloc)


def test_plan_rejects_counts_that_disagree(M):
    T, K, E, N = 10, 2, 4, 2
    idx, _ = _routing(7, T, K, E)
    counts = np.stack([np.bincount(idx[idx >= 0], minlength=E)] * N).astype(np.int32)
    counts[0, 1] += 1
    with pytest.raises(M.MMError):
        M.mm_moe_ep_plan(counts, idx, T, K, E, N, 0)
    with pytest.raises(M.MMError):                     # E not divisible by N
        M.mm_moe_ep_plan(counts[:, :3], idx % 3, T, K, 3, N, 0)


def test_plan_out_of_range_ids_are_not_sent(M):
    T, K, E, N = 6, 2, 4, 2
    idx = np.array([[0, 3], [-1, 2], [5, 1], [-3, 0], [2, 3], [1, -1]], dtype=np.int32)
    valid = (idx >= 0) & (idx < E)
    counts = np.stack([np.bincount(idx[valid], minlength=E), np.zeros(E, int)]).astype(np.int32)
    send_row, nrows, _ = M.mm_moe_ep_plan(counts, idx, T, K, E, N, 0)
    assert np.all(send_row.reshape(T, K)[~valid] == -1)
    assert np.all(send_row.reshape(T, K)[valid] >= 0)


# ------------------------------------------------------------------ two gloo ranks
def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, N, port, q):
    try:
        import torch.distributed as dist
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=N)
        from moe_expert_forward_gb300 import ep
        T, K, E = 29, 4, 8
        idx, w = _routing(200 + rank, T, K, E)
        counts_all, send_row, rows, rex = ep.plan_distributed(idx, E)
        # the metadata push of the device path, here as a gather of every rank's
        # (owner, row, pair, weight bits) list
        Eloc = E // N
        valid = send_row >= 0
        owner = np.where(valid, idx.reshape(-1) // Eloc, -1)
        mine = np.stack([owner, send_row, np.arange(T * K), w.reshape(-1).view(np.int32)], 1)[valid]
        n = torch.tensor([len(mine)])
        ns = [torch.zeros_like(n) for _ in range(N)]
        dist.all_gather(ns, n)
        cap = int(max(int(v) for v in ns))
        pad = np.full((cap, 4), -1, np.int32)
        pad[:len(mine)] = mine
        parts = [torch.empty(cap, 4, dtype=torch.int32) for _ in range(N)]
        dist.all_gather(parts, torch.from_numpy(pad))
        meta = np.full((rows, 4), -7, np.int32)
        for src, (part, cnt) in enumerate(zip(parts, ns)):
            for o, row, pair, wb in part.numpy()[:int(cnt)]:
                if o == rank:
                    meta[row] = (src, pair, -1, wb)
        q.put((rank, idx, w, counts_all, send_row, rows, rex, meta))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # reported to the parent
        q.put((rank, repr(e)))


def test_two_gloo_ranks_exchange_counts_and_metadata(M):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    N, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, N, port, q)) for r in range(N)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(N):
        item = q.get(timeout=120)
        assert len(item) > 2, item
        res[item[0]] = item[1:]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    T, K, E = 29, 4, 8
    Eloc = E // N
    idx_all = np.concatenate([res[r][0] for r in range(N)])
    w_all = np.concatenate([res[r][1] for r in range(N)])
    r, first, send, rows = _expected(idx_all, T, K, E, N)
    for rank in range(N):
        _, _, counts_all, send_row, nrows, rex, meta = res[rank]
        assert np.array_equal(counts_all[rank], np.bincount(res[rank][0][res[rank][0] >= 0], minlength=E))
        assert np.array_equal(send_row, send[rank * T:(rank + 1) * T].reshape(-1))
        assert nrows == rows[rank]
        # each received row names the right source pair (global pair = the oracle's src)
        gpair = (meta[:, 0] * T + meta[:, 1] // K) * K + meta[:, 1] % K
        assert np.array_equal(gpair, r["src"][first[rank] + np.arange(nrows)])
        assert np.array_equal(rex, idx_all.reshape(-1)[gpair] - rank * Eloc)
        assert np.array_equal(meta[:, 3].view(np.float32), w_all.reshape(-1)[gpair])


def test_recv_capacity_bounds_every_routing(M):
    """num_tokens_bound: N * bound * min(K, E/N) rows cover the worst routing (every
    token of every rank picks as many of one rank's experts as it can); the plan
    refuses a receive count above the capacity it is given."""
    assert M.mm_moe_ep_recv_capacity(64, 6, 256, 8) == 8 * 64 * 6
    assert M.mm_moe_ep_recv_capacity(64, 6, 16, 8) == 8 * 64 * 2       # 2 experts a rank
    N, T, K, E = 2, 16, 3, 8
    Eloc = E // N
    worst = [np.tile(np.arange(K, dtype=np.int32), (T, 1)) for _ in range(N)]   # all pairs to rank 0
    counts_all = np.stack([np.bincount(w.reshape(-1), minlength=E) for w in worst]).astype(np.int32)
    cap = M.mm_moe_ep_recv_capacity(T, K, E, N)
    _, rows, _ = M.mm_moe_ep_plan(counts_all, worst[0], T, K, E, N, 0, recv_capacity=cap)
    assert rows == N * T * K == cap                      # K <= E/N: the bound is reached
    small = M.mm_moe_ep_recv_capacity(T // 2, K, E, N)  # a bound below the ranks' token counts
    with pytest.raises(M.MMError):
        M.mm_moe_ep_plan(counts_all, worst[0], T, K, E, N, 0, recv_capacity=small)
