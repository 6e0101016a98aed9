"""Edge cases of the forward against the oracle: an empty batch, fully masked
routing, top-k equal to the number of experts, the largest expert count and the
largest top-k the library accepts, in both GEMM paths (fused stream and two
launches), and in the FP8 variant."""
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


def _opt(M, cfg, **kw):
    return M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8, **kw)


def _check_all_rows(M, cfg, inp, opt):
    dev = to_dev(inp)
    out, ws, _, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, f"device status {code} at site {where}"
    ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False)
    return check_output(out.float().cpu().numpy(), ref, cfg.name)


MODES = [dict(fused=1), dict(fused=0)]


@pytest.mark.parametrize("variant", ["mx", "f8"])
def test_empty_batch(M, variant):
    """T = 0: the call succeeds and launches nothing that touches a token."""
    cfg = W.Config("empty", T=0, H=256, I=128 if variant == "mx" else 256, E=4, K=2, variant=variant, seed=31)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    for kw in (MODES if variant == "mx" else [dict()]):
        out, ws, _, (code, where) = run_forward(M, cfg, dev, _opt(M, cfg, **kw))
        assert code == 0 and out.shape == (0, cfg.H), (kw, code, where)


@pytest.mark.parametrize("variant", ["mx", "f8"])
def test_all_routing_masked_gives_zeros(M, variant):
    cfg = W.Config("masked", T=50, H=256, I=128 if variant == "mx" else 256, E=6, K=3, variant=variant, seed=32)
    inp = W.make_inputs(cfg, "cpu")
    inp["topk_idx"].fill_(-1)
    dev = to_dev(inp)
    for kw in (MODES if variant == "mx" else [dict()]):
        out, ws, _, (code, where) = run_forward(M, cfg, dev, _opt(M, cfg, **kw))
        assert code == 0, (kw, code, where)
        assert torch.count_nonzero(out.float()).item() == 0, kw


@pytest.mark.parametrize("kw", MODES, ids=["fused", "two-launch"])
def test_topk_equals_experts(M, kw):
    """Every token goes to every expert: each expert gets all T rows (two blocks here)."""
    cfg = W.Config("k_eq_e", T=160, H=256, I=256, E=4, K=4, seed=33)
    _check_all_rows(M, cfg, W.make_inputs(cfg, "cpu"), _opt(M, cfg, **kw))


@pytest.mark.parametrize("kw", MODES, ids=["fused", "two-launch"])
def test_largest_expert_count(M, kw):
    """E = 1024 (the largest the library takes): most experts get no token, the
    shared-memory tables are at their largest, and the default lag (E) is the largest."""
    cfg = W.Config("e1024", T=96, H=256, I=128, E=1024, K=4, seed=34)
    _check_all_rows(M, cfg, W.make_inputs(cfg, "cpu"), _opt(M, cfg, **kw))


@pytest.mark.parametrize("variant", ["mx", "f8"])
def test_largest_topk(M, variant):
    cfg = W.Config("k16", T=40, H=256, I=256, E=32, K=16, variant=variant, seed=35)
    _check_all_rows(M, cfg, W.make_inputs(cfg, "cpu"), _opt(M, cfg))
