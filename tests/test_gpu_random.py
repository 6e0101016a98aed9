"""A seeded sweep of random shapes through every GEMM path against the oracle:
T, H, I, E, K and the routing (uniform or Zipf, with masked slots) drawn per
case, each run through the MX fused stream, the MX two-launch path and the FP8
variant, all rows compared; plus the smallest shapes the library takes and
the largest contraction the FP8 variant takes."""
import numpy as np
import pytest
import torch

import workload as W
from gpu_util import check_output, intermediate_match, oracle_rows, read_routing, run_forward, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


def _random_config(i: int) -> W.Config:
    rng = np.random.default_rng(1000 + i)
    E = int(rng.integers(1, 41))
    K = int(rng.integers(1, min(E, 8) + 1))
    return W.Config(f"rand{i}", T=int(rng.integers(1, 201)), H=128 * int(rng.integers(1, 9)),
                    I=128 * int(rng.integers(1, 9)), E=E, K=K, seed=2000 + i,
                    routing="zipf" if i % 3 == 2 else "uniform")


def _inputs(cfg, mask_frac):
    inp = W.make_inputs(cfg, "cpu")
    if mask_frac > 0:
        g = torch.Generator().manual_seed(cfg.seed)
        inp["topk_idx"][torch.rand(inp["topk_idx"].shape, generator=g) < mask_frac] = -1
    return inp


def _check(M, cfg, inp, **kw):
    dev = to_dev(inp)
    opt = M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8, **kw)
    out, ws, _, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, (cfg, kw, code, where)
    ref, inter = oracle_rows(cfg, dev, np.arange(cfg.T))
    check_output(out.float().cpu().numpy(), ref, f"{cfg} {kw}")
    _, _, slot, _, _ = read_routing(M, cfg, ws, opt)
    assert intermediate_match(M, cfg, ws, opt, slot, inter) >= 0.999


PATHS = [("mx", dict(fused=1)), ("mx", dict(fused=0)), ("f8", dict())]


@pytest.mark.parametrize("i", range(14))
def test_random_shapes_every_path(M, i):
    base = _random_config(i)
    mask = 0.1 if i % 2 else 0.0
    for variant, kw in PATHS:
        cfg = base.with_(variant=variant)
        _check(M, cfg, _inputs(cfg, mask), **kw)


@pytest.mark.parametrize("variant,kw", PATHS, ids=["mx-fused", "mx-two-launch", "f8"])
def test_smallest_shapes(M, variant, kw):
    for cfg in (W.Config("min", T=1, H=128, I=128, E=1, K=1, variant=variant, seed=51),
                W.Config("min2", T=3, H=128, I=128, E=2, K=2, variant=variant, seed=52)):
        _check(M, cfg, _inputs(cfg, 0.0), **kw)


def test_f8_long_contraction(M):
    """H = I = 8192 and H = 12288: 64 and 96 k-blocks of promotion per task."""
    cfg = W.Config("f8_big", T=16, H=8192, I=8192, E=1, K=1, variant="f8", seed=53)
    _check(M, cfg, _inputs(cfg, 0.0))
    cfg = W.Config("f8_bigger", T=16, H=12288, I=1024, E=2, K=1, variant="f8", seed=54)
    _check(M, cfg, _inputs(cfg, 0.0))
