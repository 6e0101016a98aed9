"""The two SwiGLU forms of the L1 epilogue: the fast-math form (default;
__expf and an approximate reciprocal) and the precise form (expf and the IEEE
division), each against the oracle's exact SiLU, in both variants."""
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


def _opt(M, cfg, **kw):
    return M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8, **kw)


CASES = [
    (W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), dict(fused=1)),
    (W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), dict(fused=0)),
    (W.Config("f8_ragged", T=300, H=512, I=384, E=5, K=2, variant="f8", seed=25), dict()),
]


@pytest.mark.parametrize("precise", [0, 1])
@pytest.mark.parametrize("cfg,kw", CASES, ids=["fused", "two-launch", "f8"])
def test_swiglu_form_matches_oracle(M, cfg, kw, precise):
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    opt = _opt(M, cfg, precise_swiglu=precise, **kw)
    out, ws, _, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, (code, where)
    ref, inter = oracle_rows(cfg, dev, np.arange(cfg.T))
    check_output(out.float().cpu().numpy(), ref, f"{cfg.name} precise={precise}")
    _, _, slot, _, _ = read_routing(M, cfg, ws, opt)
    assert intermediate_match(M, cfg, ws, opt, slot, inter) >= 0.999


@pytest.mark.parametrize("variant", ["mx", "f8"])
def test_fast_and_precise_forms_agree(M, variant):
    """The two forms differ by a few ulps of fp32 before the FP8 requant, so
    the outputs differ by far less than the quantisation step."""
    cfg = W.Config("k2", T=256, H=512, I=256, E=4, K=2, variant=variant, seed=44)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    a, _, prep, sa = run_forward(M, cfg, dev, _opt(M, cfg))
    a = a.float().clone()
    b, _, _, sb = run_forward(M, cfg, dev, _opt(M, cfg, precise_swiglu=1), prepared=prep)
    assert sa[0] == 0 and sb[0] == 0
    b = b.float()
    rms = a.pow(2).mean(dim=1, keepdim=True).sqrt()
    assert torch.all((a - b).abs() <= 1e-2 * rms + 1e-6)
    assert (a == b).float().mean().item() > 0.9
