"""Expert parallelism, device side: N ranks whose buffers all live on one GPU,
run step by step (count, plan, push metadata, pull rows, local forward, combine)
through the library's EP entry points.  Each rank's output equals the oracle's
bf16-partials forward of its tokens (the pages' combine receives every pair's
output as bf16) and, bit for bit, the single-GPU forward with bf16 partials over
all ranks' tokens together."""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from gpu_util import check_output, oracle_rows, run_forward, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


def _run(M, cfg, N, mask=0.0, all_to_rank0=False, combine="push", bound=None):
    from moe_expert_forward_gb300 import ep
    inp = W.make_inputs(cfg, "cpu")                     # all ranks' tokens, rank-major
    g = torch.Generator().manual_seed(cfg.seed)
    if mask:
        inp["topk_idx"][torch.rand(cfg.T, cfg.K, generator=g) < mask] = -1
    if all_to_rank0:                                    # rank 1.. own experts nobody routes to
        Eloc = cfg.E // N
        inp["topk_idx"] = torch.where(inp["topk_idx"] >= 0, inp["topk_idx"] % Eloc, inp["topk_idx"])
    dev = to_dev(inp)
    Tr = cfg.T // N
    variant = M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8
    states = [ep.RankState(r, dev["x"][r * Tr:(r + 1) * Tr].contiguous(), dev["x_sf"][r * Tr:(r + 1) * Tr].contiguous(),
                           dev["topk_idx"][r * Tr:(r + 1) * Tr].contiguous(),
                           dev["topk_w"][r * Tr:(r + 1) * Tr].contiguous(), cfg.E, N, variant) for r in range(N)]
    outs, plans = ep.forward_on_one_device(states, dev["w1"], dev["w1_sf"], dev["w2"], dev["w2_sf"], cfg.I,
                                           combine=combine, num_tokens_bound=bound)
    got = torch.cat(outs)
    # single GPU, bf16 partials, all tokens together
    single, _, _, (code, _) = run_forward(M, cfg, dev, M.options(variant, partials_bf16=1))
    assert code == 0
    return got, single, dev, plans


CFGS = [W.Config("ep_mx", T=192, H=512, I=256, E=8, K=3, seed=81),
        W.Config("ep_f8", T=128, H=512, I=256, E=8, K=2, variant="f8", seed=82)]


@pytest.mark.parametrize("N", [2, 4])
@pytest.mark.parametrize("cfg", CFGS, ids=[c.name for c in CFGS])
def test_ep_matches_oracle_and_single_gpu(M, cfg, N):
    got, single, dev, _ = _run(M, cfg, N)
    ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False, partials_bf16=True)
    check_output(got.float().cpu().numpy(), ref, f"{cfg.name} EP x{N}")
    assert torch.equal(got, single)


@pytest.mark.parametrize("N", [2, 4])
def test_ep_pull_combine_equals_push(M, N):
    """The pull form of the combine (each rank reads its slots from the owners) and
    receive buffers sized by the token bound give the same bits as the push form."""
    cfg = CFGS[0].with_(seed=84)
    got_pull, single, _, _ = _run(M, cfg, N, combine="pull", bound=cfg.T // N)
    got_push, _, _, _ = _run(M, cfg, N, combine="push")
    assert torch.equal(got_pull, got_push) and torch.equal(got_push, single)


def test_ep_masked_slots_and_idle_ranks(M):
    """Masked slots, and ranks 1..3 owning experts no token picks (they receive
    nothing and run no local forward)."""
    cfg = CFGS[0].with_(seed=83)
    got, single, dev, plans = _run(M, cfg, 4, mask=0.2, all_to_rank0=True)
    assert plans[0][1] > 0 and all(p[1] == 0 for p in plans[1:])
    assert torch.equal(got, single)
    ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False, partials_bf16=True)
    check_output(got.float().cpu().numpy(), ref, "EP idle ranks")


def test_ep_flash_shape(M):
    """The flash shape (H=4096, I=2048, E=256, top-6) split over 2 ranks of 1024
    tokens: bit for bit the single-GPU bf16-partials forward."""
    cfg = W.CONFIGS["flash"]
    got, single, _, _ = _run(M, cfg, 2)
    assert torch.equal(got, single)


def _flags(N):
    """N ranks' flag arrays (uint32 [N] each, zeroed) and the device table of them."""
    from moe_expert_forward_gb300 import ep
    arrays = [torch.zeros(N, dtype=torch.int32, device="cuda") for _ in range(N)]
    return arrays, ep.pointer_table(arrays, "cuda")


@pytest.mark.parametrize("N", [2, 4, 8])
def test_ep_barrier_all_ranks_arrive(M, N):
    """All ranks' barriers in one cooperative launch (block r is rank r): every
    flag reaches each epoch in turn and no wait runs out."""
    arrays, table = _flags(N)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for epoch in (1, 2, 3):
        assert M.mm_moe_ep_barrier_ranks(table.data_ptr(), N, epoch, 2000, 0, status.data_ptr(), s) == 0
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        assert all(torch.all(a == epoch) for a in arrays)


def test_ep_barrier_missing_rank_times_out(M):
    """Rank 2 of 4 never arrives: the others' waits run out after the deadline and
    report MM_MOE_ERR_TIMEOUT at site 301, naming rank 2; the context stays usable."""
    N = 4
    arrays, table = _flags(N)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert M.mm_moe_ep_barrier_ranks(table.data_ptr(), N, 1, 50, 1 << 2, status.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert int(status[0]) == M.MM_MOE_ERR_TIMEOUT and int(status[1]) == 301 and int(status[2]) == 2
    status.zero_()
    assert M.mm_moe_ep_barrier_ranks(table.data_ptr(), N, 2, 2000, 0, status.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert int(status[0]) == 0


def test_ep_barrier_single_rank(M):
    """The per-rank entry point with one rank: its own arrival completes it."""
    arrays, table = _flags(1)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert M.mm_moe_ep_barrier(table.data_ptr(), 1, 0, 5, 100, status.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert int(status[0]) == 0 and int(arrays[0][0]) == 5
