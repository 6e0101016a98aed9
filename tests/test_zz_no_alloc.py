"""The allocation-free routing entry point (mm_moe_dispatch_noalloc).

Some callers cannot give the library scratch memory: their runtime owns all
device memory, or an allocation on their path could synchronise the device.
This file checks, through the C ABI, that the entry point made for them gives
exactly the routing of mm_moe_dispatch (which uses caller scratch), on two
calls in a row with different routings, so a stale shared scratch would show.
It is collected last so that a stop-at-first-failure run has already run the
rest of the suite.
"""
import numpy as np
import pytest
import torch

import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


def _buffers(T, K, E, block):
    cap = T * K + min(T * K, E) * (block - 1) + 1
    return (torch.full((E,), -7, dtype=torch.int32, device="cuda"),
            torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.full((max(T * K, 1),), -7, dtype=torch.int32, device="cuda"),
            torch.full((cap,), -7, dtype=torch.int32, device="cuda"),
            torch.zeros(4, dtype=torch.int32, device="cuda"), cap)


def _route(M, idx: torch.Tensor, E: int, block: int, noalloc: bool):
    T, K = idx.shape
    cnt, blk, slot, src, status, cap = _buffers(T, K, E, block)
    stream = torch.cuda.current_stream().cuda_stream
    if noalloc:
        r = M.mm_moe_dispatch_noalloc(idx.data_ptr(), T, K, E, block, cnt.data_ptr(), blk.data_ptr(),
                                      slot.data_ptr(), src.data_ptr(), cap, status.data_ptr(), stream)
    else:
        n = M.mm_moe_dispatch_scratch_size(T, K, E)
        scratch = torch.empty(n, dtype=torch.uint8, device="cuda")
        r = M.mm_moe_dispatch(idx.data_ptr(), T, K, E, block, cnt.data_ptr(), blk.data_ptr(), slot.data_ptr(),
                              src.data_ptr(), cap, scratch.data_ptr(), n, status.data_ptr(), stream)
    assert r == M.MM_MOE_OK
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (cnt, blk, slot, src, status)]


def test_noalloc_dispatch_matches_scratch_dispatch_twice(M):
    first = W.CONFIGS["flash"]
    second = W.CONFIGS["decode"].with_(E=256)
    for cfg in (first, second):           # two calls in a row, different routing and sizes
        idx, _ = W.make_routing(cfg, "cuda")
        got = _route(M, idx, cfg.E, 128, noalloc=True)
        ref = _route(M, idx, cfg.E, 128, noalloc=False)
        for a, b in zip(got, ref):
            assert np.array_equal(a, b)
        assert got[4][0] == 0


def test_noalloc_dispatch_largest_expert_count(M):
    """1024 experts and 2^19 pairs: the fixed array holds counts for 64 CTAs,
    fewer than mm_moe_dispatch spreads this over; the routing is the same."""
    T, K, E = 65536, 8, 1024
    g = torch.Generator(device="cuda").manual_seed(5)
    idx = torch.randint(0, E, (T, K), generator=g, device="cuda", dtype=torch.int32)
    idx[torch.rand(T, K, generator=g, device="cuda") < 0.02] = -1
    got = _route(M, idx, E, 128, noalloc=True)
    ref = _route(M, idx, E, 128, noalloc=False)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)
    assert got[4][0] == 0
