"""The forward inside a CUDA graph: mm_moe_forward allocates nothing and never
synchronises, so a captured forward replays with the same results as the eager
call, in both variants, the fused stream (also with the intermediate ring) and
the two-launch path."""
import pytest
import torch

import workload as W
from gpu_util import run_forward, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


CASES = [(W.Config("g_mx", T=300, H=512, I=384, E=5, K=2, seed=91), dict(fused=1)),
         (W.Config("g_mx", T=300, H=512, I=384, E=5, K=2, seed=91), dict(fused=0)),
         (W.Config("g_f8", T=200, H=512, I=256, E=6, K=2, variant="f8", seed=92), dict()),
         # the ring's lag is chosen on the device from each replay's routing
         (W.Config("g_ring", T=256, H=256, I=256, E=64, K=6, seed=93), dict(fused=1, ring_blocks=5))]


@pytest.mark.parametrize("cfg,kw", CASES, ids=["mx_fused", "mx_two_launch", "f8", "mx_ring"])
def test_forward_replays_from_a_cuda_graph(M, cfg, kw):
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    opt = M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8, **kw)
    ref, ws, prep, (code, _) = run_forward(M, cfg, dev, opt)   # eager, also configures the kernels
    assert code == 0
    ref = ref.clone()
    out = torch.zeros_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        M.forward(dev["x"], dev["x_sf"], dev["topk_idx"], dev["topk_w"], dev["w1"], prep[0], dev["w2"], prep[1],
                  out, cfg.H, cfg.I, cfg.E, ws, opt, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert M.sync_status(ws)[0] == 0
        assert torch.equal(out, ref)
    # new inputs written into the captured buffers are picked up by the replay
    idx2 = torch.roll(dev["topk_idx"], 1, 0)
    dev["topk_idx"].copy_(idx2)
    g.replay()
    torch.cuda.synchronize()
    ref2, _, _, _ = run_forward(M, cfg, dev, opt, prepared=prep)
    assert torch.equal(out, ref2)
