"""The bf16-partials combine (each slot's L2 output cast to bf16 before the
fixed-order top-k sum) against the oracle's reading of it, in both variants and
both GEMM paths, at a full-size workload, and one exact invariant."""
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


CASES = [
    (W.CONFIGS["tiny"], dict(fused=1)),
    (W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), dict(fused=1)),
    (W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), dict(fused=0)),
    (W.Config("f8_ragged", T=300, H=512, I=384, E=5, K=2, variant="f8", seed=25), dict()),
]


@pytest.mark.parametrize("cfg,kw", CASES, ids=["tiny", "ragged-fused", "ragged-two-launch", "f8"])
def test_bf16_partials_match_oracle(M, cfg, kw):
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    out, ws, _, (code, where) = run_forward(M, cfg, dev, _opt(M, cfg, partials_bf16=1, **kw))
    assert code == 0, (code, where)
    ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False, partials_bf16=True)
    check_output(out.float().cpu().numpy(), ref, f"{cfg.name} bf16 partials")


def test_bf16_partials_fullsize_flash(M):
    cfg = W.CONFIGS["flash"]
    dev = W.make_inputs(cfg, "cuda")
    out, ws, _, (code, where) = run_forward(M, cfg, dev, _opt(M, cfg, partials_bf16=1))
    assert code == 0, (code, where)
    rows = W.eval_rows(cfg)
    ref, _ = oracle_rows(cfg, dev, rows, keep_intermediate=False, partials_bf16=True)
    check_output(out[torch.from_numpy(rows).cuda()].float().cpu().numpy(), ref, "flash bf16 partials")


@pytest.mark.parametrize("variant", ["mx", "f8"])
def test_single_slot_bf16_partials_equal_fp32_partials(M, variant):
    """With one slot per token the combine has one term, so casting that term
    to bf16 first changes nothing: bf16(bf16(y)) = bf16(y), bit for bit."""
    cfg = W.Config("k1", T=77, H=384, I=256, E=3, K=1, variant=variant, seed=42)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    a, _, prep, sa = run_forward(M, cfg, dev, _opt(M, cfg))
    a = a.clone()
    b, _, _, sb = run_forward(M, cfg, dev, _opt(M, cfg, partials_bf16=1), prepared=prep)
    assert sa[0] == 0 and sb[0] == 0
    assert torch.equal(a, b)
