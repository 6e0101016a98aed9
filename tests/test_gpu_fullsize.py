"""Parity at the workload sizes the benchmark times (flash, pro, decode), in the
launch configuration bench.py uses: every output row of a seeded sample is
checked against the oracle, the routing is checked in full, and the sampled
rows' intermediate codes are compared."""
import gc

import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from gpu_util import check_output, intermediate_match, oracle_rows, read_routing, run_forward

pytestmark = pytest.mark.gpu

SAMPLE_ROWS = {"flash": 8, "pro": 4, "decode": 12, "f8": 4}


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


@pytest.mark.parametrize("name,fused", [("flash", 0), ("flash", 1), ("decode", 1), ("pro", 1), ("pro", 0), ("f8", 0)])
def test_fullsize_sampled_rows(M, name, fused):
    cfg = W.CONFIGS[name]
    dev = W.make_inputs(cfg, "cuda")
    opt = M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8, fused=fused)
    out, ws, prepared, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, f"device status {code} at site {where}"
    cnt, blk, slot, src, bm = read_routing(M, cfg, ws, opt)
    ref_route = O.route(dev["topk_idx"].cpu().numpy(), cfg.E, bm)
    assert np.array_equal(cnt, ref_route["cnt"]) and np.array_equal(blk, ref_route["blk_off"])
    assert np.array_equal(slot, ref_route["slot"])
    rows = W.eval_rows(cfg)
    rng = np.random.default_rng(cfg.seed + 11)
    rows = np.sort(rng.choice(rows, min(SAMPLE_ROWS[name], len(rows)), replace=False))
    ref, inter = oracle_rows(cfg, dev, rows)
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    check_output(got, ref, name)
    assert intermediate_match(M, cfg, ws, opt, slot, inter) >= 0.999
    # whole-output properties: finite, and every token that has an expert is non-zero
    assert torch.isfinite(out.float()).all()
    del dev, out, ws, prepared
    gc.collect()
    torch.cuda.empty_cache()
