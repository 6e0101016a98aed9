"""The fused stream's early combine (epilogue warps reduce the tokens whose
experts have finished L2, instead of a combine launch after the GEMM) gives
the combine kernel's bits, with fp32 and bf16 partials, with
masked slots, many empty experts and the largest top-k, and at full size; it
is also checked against the oracle through every other fused-path test, which
run with it on (the default)."""
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


def _both(M, cfg, dev, **kw):
    opt = lambda ec: M.options(M.MM_MOE_VARIANT_MX, fused=1, early_combine=ec, **kw)
    a, _, prep, sa = run_forward(M, cfg, dev, opt(1))
    assert sa[0] == 0, sa
    a = a.clone()
    b, _, _, sb = run_forward(M, cfg, dev, opt(0), prepared=prep)
    assert sb[0] == 0, sb
    return a, b


def _masked(cfg):
    inp = W.make_inputs(cfg, "cpu")
    g = torch.Generator().manual_seed(cfg.seed)
    inp["topk_idx"][torch.rand(inp["topk_idx"].shape, generator=g) < 0.2] = -1
    return inp


CASES = [
    ("tiny", W.CONFIGS["tiny"], {}, None),
    ("ragged", W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), {}, None),
    ("ragged-bf16-partials", W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), {"partials_bf16": 1}, None),
    ("k3", W.Config("k3", T=120, H=384, I=256, E=6, K=3, seed=41), {}, None),
    ("masked", W.Config("masked", T=200, H=256, I=256, E=8, K=4, seed=48), {}, _masked),
    ("e1024", W.Config("e1024", T=96, H=256, I=128, E=1024, K=4, seed=34), {}, None),
    ("k16", W.Config("k16", T=40, H=256, I=256, E=32, K=16, seed=35), {}, None),
]


@pytest.mark.parametrize("name,cfg,kw,make", CASES, ids=[c[0] for c in CASES])
def test_early_combine_bits_equal_combine_kernel(M, name, cfg, kw, make):
    dev = to_dev(make(cfg) if make else W.make_inputs(cfg, "cpu"))
    a, b = _both(M, cfg, dev, **kw)
    assert torch.equal(a, b)
    ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False,
                         partials_bf16=bool(kw.get("partials_bf16")))
    check_output(a.float().cpu().numpy(), ref, f"{name} early combine")


@pytest.mark.parametrize("name", ["flash", "decode"])
def test_early_combine_fullsize_bits(M, name):
    cfg = W.CONFIGS[name]
    dev = W.make_inputs(cfg, "cuda")
    a, b = _both(M, cfg, dev)
    assert torch.equal(a, b)
