"""Device-side failure detection without faulting the GPU: a wait that nothing
will ever satisfy must end with MM_MOE_ERR_TIMEOUT after the deadline, and the
CUDA context must stay usable."""
import time

import numpy as np
import pytest
import torch

import workload as W
from gpu_util import check_output, oracle_rows, run_forward, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


def test_unreachable_wait_times_out_and_context_survives(M):
    cfg = W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    opt = M.options(fused=1, debug_flags=4, wait_timeout_ms=50)
    t0 = time.time()
    out, ws, prep, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == M.MM_MOE_ERR_TIMEOUT
    # the first deadline to pass is either the producer's wait for the block's L1
    # tiles (106) or the MMA issuer's wait for the stage that producer never fills (102)
    assert where in (102, 106), where
    assert time.time() - t0 < 30
    # the next call on the same context and workspace is correct
    out2, ws2, _, (code2, _) = run_forward(M, cfg, dev, M.options(fused=1), ws=ws, prepared=prep)
    assert code2 == 0
    ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False)
    check_output(out2.float().cpu().numpy(), ref, "after timeout")


@pytest.mark.parametrize("bad", [11, -2, -7])
def test_bad_routing_is_reported(M, bad):
    """Expert ids >= E or < -1 are masked (the slot contributes nothing) and flagged."""
    cfg = W.Config("tiny", T=64, H=256, I=128, E=8, K=2, seed=3)
    inp = W.make_inputs(cfg, "cpu")
    inp["topk_idx"][5, 1] = bad
    dev = to_dev(inp)
    out, ws, prep, (code, where) = run_forward(M, cfg, dev)
    assert code == M.MM_MOE_ERR_BAD_ROUTING
    # the flagged slot is masked exactly as -1 would be
    masked = {k: v.clone() for k, v in dev.items()}
    masked["topk_idx"][5, 1] = -1
    out_m, _, _, (code_m, _) = run_forward(M, cfg, masked, prepared=prep)
    assert code_m == 0 and torch.equal(out, out_m)


def test_host_rejections(M):
    cfg = W.CONFIGS["tiny"]
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    opt = M.options()
    w1p, w2p = M.prepare_weights(dev["w1_sf"], dev["w2_sf"], cfg.H, cfg.I, cfg.E, opt)
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(M.MMError) as ei:
        M.forward(dev["x"], dev["x_sf"], dev["topk_idx"], dev["topk_w"], dev["w1"], w1p, dev["w2"], w2p, out,
                  cfg.H, cfg.I, cfg.E, small, opt)
    assert ei.value.code == M.MM_MOE_ERR_WORKSPACE_TOO_SMALL
    ws = M.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, opt)
    with pytest.raises(M.MMError) as ei:                   # misaligned weights
        M.forward(dev["x"], dev["x_sf"], dev["topk_idx"], dev["topk_w"], dev["w1"].view(-1)[1:], w1p, dev["w2"],
                  w2p, out, cfg.H, cfg.I, cfg.E, ws, opt)
    assert ei.value.code == M.MM_MOE_ERR_INVALID_ARG


def test_f8_unreachable_wait_times_out_and_context_survives(M):
    """FP8: the last stage of every CTA's last L1 task is never loaded.  The issuer's
    wait for it runs out, the abort reaches the commit waiter, the epilogue and
    the other issuer through their named barriers (every phase keeps its count),
    and the next call on the same context is correct."""
    cfg = W.Config("f8_ragged", T=300, H=512, I=384, E=5, K=2, variant="f8", seed=25)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    opt = M.options(M.MM_MOE_VARIANT_F8, debug_flags=4, wait_timeout_ms=50)
    t0 = time.time()
    out, ws, prep, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == M.MM_MOE_ERR_TIMEOUT
    # the first deadline to pass is the issuer's wait for the stage that is never
    # loaded (202) or the commit waiter's wait for that unit's MMAs (204)
    assert where in (202, 204), where
    assert time.time() - t0 < 30
    out2, _, _, (code2, _) = run_forward(M, cfg, dev, M.options(M.MM_MOE_VARIANT_F8), ws=ws, prepared=prep)
    assert code2 == 0
    ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False)
    check_output(out2.float().cpu().numpy(), ref, "FP8 after timeout")
