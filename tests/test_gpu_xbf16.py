"""bf16 activations quantised inside the gather (Options.x_bf16): the pool the
GEMMs read must be exactly the one the e4m3 path builds from the oracle's
quantisation of the same rows, so the outputs are bit-identical to feeding the
oracle's codes and scales, in both variants and both MX GEMM paths; and the
outputs match the oracle's forward on those codes."""
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


def _opt(M, cfg, **kw):
    return M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8, **kw)


def _oracle_quantised(cfg, xb: torch.Tensor, device):
    codes, sf = O.quantise_x(xb.float().cpu().numpy(), cfg.variant)
    return torch.from_numpy(codes).to(device), torch.from_numpy(np.ascontiguousarray(sf)).to(device)


def _pair(M, cfg, dev, xb, **kw):
    """(out with bf16 x, out with the oracle's codes of the same x), one prepared weight set."""
    bdev = dict(dev, x=xb, x_sf=None)
    a, _, prep, sa = run_forward(M, cfg, bdev, _opt(M, cfg, x_bf16=1, **kw))
    assert sa[0] == 0, sa
    a = a.clone()
    qx, qsf = _oracle_quantised(cfg, xb, "cuda")
    qdev = dict(dev, x=qx, x_sf=qsf)
    b, _, _, sb = run_forward(M, cfg, qdev, _opt(M, cfg, **kw), prepared=prep)
    assert sb[0] == 0, sb
    return a, b, qdev


CASES = [
    (W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), dict(fused=1)),
    (W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), dict(fused=0)),
    (W.Config("f8_ragged", T=300, H=512, I=384, E=5, K=2, variant="f8", seed=25), dict()),
]


@pytest.mark.parametrize("cfg,kw", CASES, ids=["fused", "two-launch", "f8"])
def test_bf16_input_equals_oracle_quantised_input(M, cfg, kw):
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    xb = W.make_x_bf16(cfg, "cpu").cuda()
    a, b, qdev = _pair(M, cfg, dev, xb, **kw)
    assert torch.equal(a, b)
    ref, _ = oracle_rows(cfg, qdev, np.arange(cfg.T), keep_intermediate=False)
    check_output(a.float().cpu().numpy(), ref, f"{cfg.name} bf16 x")


@pytest.mark.parametrize("variant", ["mx", "f8"])
def test_bf16_input_wide_dynamic_range(M, variant):
    """Rows spanning 1e-6 .. 1e4 in magnitude, zero rows and single spikes: every
    block's scale and codes still equal the oracle's (bit-identical outputs)."""
    cfg = W.Config("range", T=64, H=512, I=256, E=4, K=2, variant=variant, seed=46)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    g = torch.Generator().manual_seed(9)
    xb = torch.randn(cfg.T, cfg.H, generator=g) * torch.logspace(-6, 4, cfg.T)[:, None]
    xb[5] = 0.0
    xb[6, 17] = 3.0e4
    xb = xb.to(torch.bfloat16).cuda()
    a, b, _ = _pair(M, cfg, dev, xb)
    assert torch.equal(a, b)


def test_bf16_input_fullsize_flash(M):
    cfg = W.CONFIGS["flash"]
    dev = W.make_inputs(cfg, "cuda")
    xb = W.make_x_bf16(cfg, "cuda")
    a, b, _ = _pair(M, cfg, dev, xb)
    assert torch.equal(a, b)


def test_e4m3_input_still_requires_x_sf(M):
    """x_sf may be NULL only on the bf16 path: the e4m3 path rejects it."""
    cfg = W.Config("k2", T=16, H=256, I=128, E=2, K=2, seed=47)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    prep = M.prepare_weights(dev["w1_sf"], dev["w2_sf"], cfg.H, cfg.I, cfg.E, _opt(M, cfg))
    ws = M.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, _opt(M, cfg))
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    r = M.mm_moe_forward(dev["x"].data_ptr(), 0, dev["topk_idx"].data_ptr(), dev["topk_w"].data_ptr(),
                         dev["w1"].data_ptr(), prep[0].data_ptr(), dev["w2"].data_ptr(), prep[1].data_ptr(),
                         out.data_ptr(), cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, ws.data_ptr(), ws.numel(),
                         _opt(M, cfg), torch.cuda.current_stream().cuda_stream)
    assert r == M.MM_MOE_ERR_INVALID_ARG
