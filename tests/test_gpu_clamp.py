"""The optional activation clamp (gate and up limited to [-c, c] before the
SwiGLU) against the oracle, in both variants and every GEMM path, at a
full-size workload, and one exact invariant."""
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


# c = 0.05 clamps most pre-activations here (their spread is about 0.3 at H = 256..512)
CASES = [
    (W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), dict(fused=1)),
    (W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), dict(fused=0)),
    (W.Config("f8_ragged", T=300, H=512, I=384, E=5, K=2, variant="f8", seed=25), dict()),
]


@pytest.mark.parametrize("cfg,kw", CASES, ids=["fused", "two-launch", "f8"])
def test_activation_clamp_matches_oracle(M, cfg, kw):
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    opt = _opt(M, cfg, activation_clamp=0.05, **kw)
    out, ws, _, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, (code, where)
    rows = np.arange(cfg.T)
    ref, inter = oracle_rows(cfg, dev, rows, clamp=0.05)
    check_output(out.float().cpu().numpy(), ref, f"{cfg.name} clamp")
    _, _, slot, _, _ = read_routing(M, cfg, ws, opt)
    assert intermediate_match(M, cfg, ws, opt, slot, inter) >= 0.999


def test_activation_clamp_fullsize_flash(M):
    cfg = W.CONFIGS["flash"]
    dev = W.make_inputs(cfg, "cuda")
    out, ws, _, (code, where) = run_forward(M, cfg, dev, _opt(M, cfg, activation_clamp=0.5))
    assert code == 0, (code, where)
    rows = W.eval_rows(cfg)
    ref, _ = oracle_rows(cfg, dev, rows, keep_intermediate=False, clamp=0.5)
    check_output(out[torch.from_numpy(rows).cuda()].float().cpu().numpy(), ref, "flash clamp")


@pytest.mark.parametrize("variant", ["mx", "f8"])
def test_huge_clamp_changes_nothing(M, variant):
    cfg = W.Config("k2", T=77, H=384, I=256, E=3, K=2, variant=variant, seed=43)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    a, _, prep, sa = run_forward(M, cfg, dev, _opt(M, cfg))
    a = a.clone()
    b, _, _, sb = run_forward(M, cfg, dev, _opt(M, cfg, activation_clamp=1e30), prepared=prep)
    assert sa[0] == 0 and sb[0] == 0
    assert torch.equal(a, b)
