"""Expert parallelism over N ranks, driven through the library's EP entry points
(include/mm_moe.h, mm_moe_ep_*).

Rank r owns experts [r*E/N, (r+1)*E/N).  One forward runs, on every rank:
count -> exchange counts -> plan -> push metadata -> barrier -> pull rows ->
local forward (K = 1 over the received pairs) -> barrier -> combine
(llm-infra-atlas "07 · MegaMoE" §7 count / push metadata / pull data and §9
combine; DeepGEMM PR #440 "How it works").  The kernels read and write peers'
buffers through device tables of their addresses; the exchange of the counts and
the barriers are host collectives, so no kernel waits on another rank.

The combine comes in the pages' push form (each owner stores every received row's
bf16 output into the token's rank, which then sums its slots locally) and a pull
form (each rank reads its slots' outputs from their owners); both give the same
bits.  `plan_distributed` is the host side of a multi-process run
(torch.distributed: an all-gather of the counts).  `forward_distributed` is one
rank's whole forward in a multi-process run: the peers' buffers are mapped into
this process by CUDA IPC (`share_peers`), and a device synchronisation plus a
process-group barrier separates the steps, so no kernel ever waits for another
process.  `EPRank` is the same rank with its buffers and the peers' addresses
set up once and kept across calls (inputs copied into a bound-sized input
region each call).  `forward_on_one_device` runs N ranks whose buffers all live
in one process, step by step from the host.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

from . import (MM_MOE_VARIANT_MX, MMError, _check, alloc_workspace, forward, mm_moe_ep_combine,
               mm_moe_ep_combine_local, mm_moe_ep_count, mm_moe_ep_plan, mm_moe_ep_pull, mm_moe_ep_push_meta,
               mm_moe_ep_push_out, mm_moe_ep_recv_capacity, options, prepare_weights, sync_status)


def host_counts(topk_idx: np.ndarray, E: int) -> np.ndarray:
    """Pairs per expert of one rank's routing (ids outside [0, E) not counted)."""
    idx = np.asarray(topk_idx).reshape(-1)
    idx = idx[(idx >= 0) & (idx < E)]
    return np.bincount(idx, minlength=E).astype(np.int32)


def plan_distributed(topk_idx: np.ndarray, E: int, group=None):
    """All-gather every rank's per-expert counts, then plan this rank's pairs.
    Returns (counts_all [N, E], send_row [T*K], recv_rows, recv_expert)."""
    import torch
    import torch.distributed as dist
    N = dist.get_world_size(group)
    rank = dist.get_rank(group)
    mine = torch.from_numpy(host_counts(topk_idx, E))
    parts = [torch.empty_like(mine) for _ in range(N)]
    dist.all_gather(parts, mine, group=group)
    counts_all = torch.stack(parts).numpy()
    T, K = np.asarray(topk_idx).shape
    send_row, rows, rex = mm_moe_ep_plan(counts_all, topk_idx, T, K, E, N, rank)
    return counts_all, send_row, rows, rex


def pointer_table(tensors: Sequence, device):
    """Device int64 array of the tensors' addresses (a peer-pointer table)."""
    import torch
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=device)


class RankState:
    """One rank's buffers: its tokens, its plan and its receive buffers."""

    def __init__(self, rank: int, x, x_sf, topk_idx, topk_w, E: int, N: int, variant: int):
        self.rank, self.E, self.N, self.variant = rank, E, N, variant
        self.x, self.x_sf, self.topk_idx, self.topk_w = x, x_sf, topk_idx, topk_w
        self.T, self.K = topk_idx.shape
        self.H = x.shape[1]


def forward_on_one_device(states: List[RankState], w1, w1_sf, w2, w2_sf, I: int, opt=None, stream=None,
                          combine: str = "push", num_tokens_bound: Optional[int] = None):
    """Run the EP forward for every rank in `states` (buffers on one device).
    w1 / w1_sf / w2 / w2_sf hold all E experts in the layouts of mm_moe.h; rank r
    uses experts [r*E/N, (r+1)*E/N).  combine: "push" (the pages' form) or "pull".
    num_tokens_bound: receive buffers sized once by mm_moe_ep_recv_capacity (every
    rank's T must be within the bound).  Returns the per-rank bf16 outputs [T_r, H]
    and the per-rank plans (send_row, recv_rows, recv_expert)."""
    import torch
    N = len(states)
    E, H, variant = states[0].E, states[0].H, states[0].variant
    Eloc = E // N
    dev = states[0].x.device
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    base_opt = opt if opt is not None else options(variant)
    # 1. counts on the device, gathered on the host (the all-gather of a multi-GPU run)
    counts = []
    for st in states:
        c = torch.empty(E, dtype=torch.int32, device=dev)
        _check(mm_moe_ep_count(st.topk_idx.data_ptr(), st.T, st.K, E, c.data_ptr(), s), "mm_moe_ep_count")
        counts.append(c)
    counts_all = torch.stack(counts).cpu().numpy()
    # 2. plans and receive buffers
    plans = []
    cap = None
    if num_tokens_bound is not None:
        cap = mm_moe_ep_recv_capacity(num_tokens_bound, states[0].K, E, N)
    for st in states:
        send_row, rows, rex = mm_moe_ep_plan(counts_all, st.topk_idx.cpu().numpy(), st.T, st.K, E, N, st.rank,
                                             recv_capacity=cap)
        st.send_row = torch.from_numpy(np.ascontiguousarray(send_row)).to(dev)
        st.rows = rows
        st.meta = torch.zeros(max(rows if cap is None else cap, 1), 4, dtype=torch.int32, device=dev)
        plans.append((send_row, rows, rex))
    # 3. metadata pushed into the owners' buffers
    peer_meta = pointer_table([st.meta for st in states], dev)
    for st in states:
        _check(mm_moe_ep_push_meta(st.topk_idx.data_ptr(), st.topk_w.data_ptr(), st.send_row.data_ptr(), st.T, st.K,
                                   E, N, st.rank, peer_meta.data_ptr(), s), "mm_moe_ep_push_meta")
    torch.cuda.synchronize()                                  # barrier
    # 4. rows pulled from the source ranks, then each rank's local forward
    peer_x = pointer_table([st.x for st in states], dev)
    peer_xsf = pointer_table([st.x_sf for st in states], dev)
    sf_row = H // 32 if variant == MM_MOE_VARIANT_MX else H // 128
    sf_dtype = torch.uint8 if variant == MM_MOE_VARIANT_MX else torch.float32
    for st in states:
        R = st.rows
        st.out_recv = torch.zeros(max(R, 1), H, dtype=torch.bfloat16, device=dev)
        if R == 0:
            continue
        x_recv = torch.empty(R, H, dtype=torch.uint8, device=dev)
        xsf_recv = torch.empty(R, sf_row, dtype=sf_dtype, device=dev)
        idx_recv = torch.empty(R, 1, dtype=torch.int32, device=dev)
        w_recv = torch.empty(R, 1, dtype=torch.float32, device=dev)
        _check(mm_moe_ep_pull(st.meta.data_ptr(), R, st.K, H, variant, peer_x.data_ptr(), peer_xsf.data_ptr(),
                              x_recv.data_ptr(), xsf_recv.data_ptr(), idx_recv.data_ptr(), w_recv.data_ptr(), s),
               "mm_moe_ep_pull")
        lo, hi = st.rank * Eloc, (st.rank + 1) * Eloc
        w1p, w2p = prepare_weights(w1_sf[lo:hi].contiguous(), w2_sf[lo:hi].contiguous(), H, I, Eloc, base_opt)
        ws = alloc_workspace(R, H, I, Eloc, 1, base_opt, dev)
        forward(x_recv, xsf_recv, idx_recv, w_recv, w1[lo:hi].contiguous(), w1p, w2[lo:hi].contiguous(), w2p,
                st.out_recv, H, I, Eloc, ws, base_opt)
        code, where = sync_status(ws)
        if code != 0:
            raise MMError(code, f"rank {st.rank} local forward (site {where})")
    torch.cuda.synchronize()                                  # barrier
    # 5. combine
    outs = []
    if combine == "push":
        # each owner stores its rows' outputs at the pairs' places in the token ranks
        parts = [torch.empty(max(st.T * st.K, 1), H, dtype=torch.bfloat16, device=dev) for st in states]
        peer_part = pointer_table(parts, dev)
        for st in states:
            _check(mm_moe_ep_push_out(st.meta.data_ptr(), st.rows, H, st.out_recv.data_ptr(), peer_part.data_ptr(), s),
                   "mm_moe_ep_push_out")
        torch.cuda.synchronize()                              # barrier
        for st, part in zip(states, parts):
            out = torch.empty(st.T, H, dtype=torch.bfloat16, device=dev)
            _check(mm_moe_ep_combine_local(st.topk_idx.data_ptr(), st.T, st.K, E, H, part.data_ptr(), out.data_ptr(),
                                           s), "mm_moe_ep_combine_local")
            outs.append(out)
    else:
        peer_out = pointer_table([st.out_recv for st in states], dev)
        for st in states:
            out = torch.empty(st.T, H, dtype=torch.bfloat16, device=dev)
            _check(mm_moe_ep_combine(st.topk_idx.data_ptr(), st.send_row.data_ptr(), st.T, st.K, E, N, H,
                                     peer_out.data_ptr(), out.data_ptr(), s), "mm_moe_ep_combine")
            outs.append(out)
    torch.cuda.synchronize()
    return outs, plans


def share_peers(tensors: Sequence, group=None):
    """Every rank's copy of each tensor in `tensors`, mapped into this process.

    The handles travel through the process group (an all-gather of picklable
    objects); each peer allocation is opened with CUDA IPC by torch's own CUDA
    tensor sharing, which also keeps the producer's block alive until every
    consumer has released it.  This rank's entries are the tensors themselves.
    Returns [len(tensors)][N] tensors; drop them (and barrier) before a peer
    frees its buffers."""
    import torch.distributed as dist
    from torch.multiprocessing.reductions import rebuild_cuda_tensor, reduce_tensor
    N = dist.get_world_size(group)
    rank = dist.get_rank(group)
    import torch
    # an empty tensor (a rank without tokens) has no allocation to share, and no
    # kernel reads through its address: it travels as None and maps to an empty tensor
    mine = [reduce_tensor(t)[1] if t.numel() else None for t in tensors]
    every = [None] * N
    dist.all_gather_object(every, mine, group=group)

    def peer(r, i, t):
        if r == rank:
            return t
        h = every[r][i]
        return rebuild_cuda_tensor(*h) if h is not None else torch.empty(0, dtype=t.dtype, device=t.device)
    return [[peer(r, i, t) for r in range(N)] for i, t in enumerate(tensors)]


def forward_distributed(st: RankState, w1, w1_sf, w2, w2_sf, I: int, opt=None, group=None, combine: str = "push",
                        num_tokens_bound: Optional[int] = None):
    """One rank's EP forward in a multi-process run (one process per rank; the
    ranks may share a GPU or not): an `EPRank` sized for `num_tokens_bound` tokens
    (default: the largest rank's token count, gathered here), one call of its
    forward, and its release.  st holds this rank's tokens; w1 / w1_sf / w2 /
    w2_sf hold all E experts in the layouts of mm_moe.h.  Steps: count ->
    all-gather the counts -> plan -> push metadata -> barrier -> pull rows and the
    local forward -> barrier -> combine (push: store row outputs into the token
    ranks, barrier, local sum; pull: read the slots from their owners) ->
    barrier.  Returns this rank's bf16 output [T, H] and its plan (send_row,
    recv_rows, recv_expert).  Collective: every rank calls it together."""
    import torch.distributed as dist
    N = dist.get_world_size(group)
    if num_tokens_bound is None:
        every = [None] * N
        dist.all_gather_object(every, int(st.T), group=group)
        num_tokens_bound = max(every)
    ctx = EPRank(st.rank, N, st.E, st.K, st.H, I, st.variant, num_tokens_bound, w1, w1_sf, w2, w2_sf, st.x.device,
                 opt, group)
    try:
        return ctx.forward(st.x, st.x_sf, st.topk_idx, st.topk_w, combine=combine)
    finally:
        ctx.close()


class EPRank:
    """One rank of a multi-process EP layer whose buffers outlive its forwards,
    as the pages' symmetric buffer does (llm-infra-atlas "07 · MegaMoE" §3: one
    buffer per rank with an input region for x and its scales; DeepGEMM PR #440:
    receive space sized by `num_tokens_bound`).

    The constructor allocates, for at most `num_tokens_bound` tokens a call: the
    input region (x and its scales, which peers pull from), the metadata and row
    output buffers of the pairs this rank receives (mm_moe_ep_recv_capacity
    rows), the combine's slot buffer, and the local forward's receive rows and
    workspace; it prepares the local experts' weight scales and exchanges every
    peer-visible buffer's address once (`share_peers`, a collective: every rank
    constructs its EPRank together).  `forward` then runs the steps of
    `forward_distributed` on those buffers; every rank calls it together, each
    with its own tokens.  `close` (collective) releases the peers' mappings."""

    def __init__(self, rank: int, N: int, E: int, K: int, H: int, I: int, variant: int, num_tokens_bound: int,
                 w1, w1_sf, w2, w2_sf, device, opt=None, group=None):
        import torch
        import torch.distributed as dist
        assert dist.get_rank(group) == rank and dist.get_world_size(group) == N and E % N == 0
        self.rank, self.N, self.E, self.K, self.H, self.I, self.variant = rank, N, E, K, H, I, variant
        self.bound, self.group, self.dev = num_tokens_bound, group, device
        self.opt = opt if opt is not None else options(variant)
        self.Eloc = E // N
        self.cap = mm_moe_ep_recv_capacity(num_tokens_bound, K, E, N)
        room = max(self.cap, 1)
        B = max(num_tokens_bound, 1)
        sf_row = H // 32 if variant == MM_MOE_VARIANT_MX else H // 128
        sf_dtype = torch.uint8 if variant == MM_MOE_VARIANT_MX else torch.float32
        # peer-visible: the input region, the metadata and row outputs this rank receives, its slot buffer
        self.x_in = torch.zeros(B, H, dtype=torch.uint8, device=device)
        self.xsf_in = torch.zeros(B, sf_row, dtype=sf_dtype, device=device)
        self.meta = torch.zeros(room, 4, dtype=torch.int32, device=device)
        self.out_recv = torch.zeros(room, H, dtype=torch.bfloat16, device=device)
        self.parts = torch.zeros(B * K, H, dtype=torch.bfloat16, device=device)
        # local: the pulled rows, their K = 1 routing, the local forward's workspace and weights
        self.x_recv = torch.empty(room, H, dtype=torch.uint8, device=device)
        self.xsf_recv = torch.empty(room, sf_row, dtype=sf_dtype, device=device)
        self.idx_recv = torch.empty(room, 1, dtype=torch.int32, device=device)
        self.w_recv = torch.empty(room, 1, dtype=torch.float32, device=device)
        self.ws = alloc_workspace(room, H, I, self.Eloc, 1, self.opt, device)
        lo, hi = rank * self.Eloc, (rank + 1) * self.Eloc
        self.w1, self.w2 = w1[lo:hi].contiguous(), w2[lo:hi].contiguous()
        self.w1p, self.w2p = prepare_weights(w1_sf[lo:hi].contiguous(), w2_sf[lo:hi].contiguous(), H, I, self.Eloc,
                                             self.opt)
        self._peers = share_peers([self.meta, self.x_in, self.xsf_in, self.out_recv, self.parts], group)
        self.t_meta, self.t_x, self.t_xsf, self.t_out, self.t_part = (pointer_table(p, device) for p in self._peers)
        self._barrier()

    def _barrier(self):
        import torch
        import torch.distributed as dist
        torch.cuda.synchronize()
        dist.barrier(group=self.group)

    def forward(self, x, x_sf, topk_idx, topk_w, combine: str = "push"):
        """This rank's bf16 output [T, H] for its T <= num_tokens_bound tokens, and
        its plan (send_row, recv_rows, recv_expert)."""
        import torch
        import torch.distributed as dist
        T, K = topk_idx.shape
        assert K == self.K and T <= self.bound and x.shape == (T, self.H)
        N, E, H, rank, dev = self.N, self.E, self.H, self.rank, self.dev
        s = torch.cuda.current_stream().cuda_stream
        if T:
            self.x_in[:T].copy_(x)
            self.xsf_in[:T].copy_(x_sf)
        c = torch.empty(E, dtype=torch.int32, device=dev)
        _check(mm_moe_ep_count(topk_idx.data_ptr(), T, K, E, c.data_ptr(), s), "mm_moe_ep_count")
        every = [None] * N
        dist.all_gather_object(every, c.cpu().numpy(), group=self.group)
        send_row, rows, rex = mm_moe_ep_plan(np.stack(every), topk_idx.cpu().numpy(), T, K, E, N, rank,
                                             recv_capacity=self.cap)
        send_row_d = torch.from_numpy(np.ascontiguousarray(send_row)).to(dev)
        _check(mm_moe_ep_push_meta(topk_idx.data_ptr(), topk_w.data_ptr(), send_row_d.data_ptr(), T, K, E, N, rank,
                                   self.t_meta.data_ptr(), s), "mm_moe_ep_push_meta")
        self._barrier()
        R = rows
        if R > 0:
            _check(mm_moe_ep_pull(self.meta.data_ptr(), R, K, H, self.variant, self.t_x.data_ptr(),
                                  self.t_xsf.data_ptr(), self.x_recv.data_ptr(), self.xsf_recv.data_ptr(),
                                  self.idx_recv.data_ptr(), self.w_recv.data_ptr(), s), "mm_moe_ep_pull")
            forward(self.x_recv[:R], self.xsf_recv[:R], self.idx_recv[:R], self.w_recv[:R], self.w1, self.w1p,
                    self.w2, self.w2p, self.out_recv[:R], H, self.I, self.Eloc, self.ws, self.opt)
            code, where = sync_status(self.ws)
            if code != 0:
                raise MMError(code, f"rank {rank} local forward (site {where})")
        self._barrier()
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        if combine == "push":
            _check(mm_moe_ep_push_out(self.meta.data_ptr(), R, H, self.out_recv.data_ptr(), self.t_part.data_ptr(),
                                      s), "mm_moe_ep_push_out")
            self._barrier()
            _check(mm_moe_ep_combine_local(topk_idx.data_ptr(), T, K, E, H, self.parts.data_ptr(), out.data_ptr(),
                                           s), "mm_moe_ep_combine_local")
        else:
            _check(mm_moe_ep_combine(topk_idx.data_ptr(), send_row_d.data_ptr(), T, K, E, N, H,
                                     self.t_out.data_ptr(), out.data_ptr(), s), "mm_moe_ep_combine")
        # the next call overwrites buffers that peers read in this one
        self._barrier()
        return out, (send_row, rows, rex)

    def close(self):
        self._barrier()
        self._peers = None
        self._barrier()
