"""FP8 intermediate scale width (Options.f8_act_gran): per-64 and per-128
requantisation of the SwiGLU output, and the L2 GEMM that dequantises each
64-wide half of a 128-K step with its own scale, against the oracle; the
default follows the pages' shape rule; the fast requant division is bit-equal
to dividing every code."""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from gpu_util import (check_output, f8_gran, intermediate_match, oracle_rows, read_routing, run_forward, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


# I >= 2048 in every case: one intermediate code that lands on the other side of an
# e4m3 rounding boundary than the oracle's (the fp32 sums differ in order) moves an
# output element by about 0.07 x amax/rms(a) x |w2|/rms(w2) / sqrt(I) of its row's
# RMS, which at small I can exceed the per-element criterion by itself.
CFGS = {
    "ragged": W.Config("f8g_ragged", T=130, H=384, I=2048, E=3, K=2, variant="f8", seed=61),
    "wide": W.Config("f8g_wide", T=96, H=1024, I=2048, E=3, K=3, variant="f8", seed=62),
    "many": W.Config("f8g_many", T=64, H=512, I=2048, E=12, K=4, variant="f8", seed=63),
}


def _check(M, cfg, gran, inp=None):
    inp = inp if inp is not None else W.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    opt = M.options(M.MM_MOE_VARIANT_F8, f8_act_gran=gran)
    out, ws, prep, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, f"device status {code} at site {where}"
    _, _, slot, _, _ = read_routing(M, cfg, ws, opt)
    g = f8_gran(cfg, opt)
    ref, inter = oracle_rows(cfg, dev, np.arange(cfg.T), f8_gran=g)
    check_output(out.float().cpu().numpy(), ref, f"{cfg.name} gran {g}")
    frac = intermediate_match(M, cfg, ws, opt, slot, inter, f"{cfg.name} gran {g}")
    assert frac >= 0.999, frac
    return out.clone(), ws, opt, prep, dev


@pytest.mark.parametrize("gran", [64, 128])
@pytest.mark.parametrize("name", list(CFGS))
def test_f8_scale_width_matches_oracle(M, name, gran):
    _check(M, CFGS[name], gran)


def test_f8_shape_rule_and_default(M):
    """-1 follows the pages' shape rule (H = 384: 64; H = 1024, I = 2048: 128) and 0,
    the default, is per 128."""
    cfg = CFGS["ragged"]
    assert O.f8_act_gran(cfg.H, cfg.I) == 64
    a, *_ = _check(M, cfg, -1)
    b, *_ = _check(M, cfg, 64)
    assert torch.equal(a, b)
    cfg2 = CFGS["wide"]
    assert O.f8_act_gran(cfg2.H, cfg2.I) == 128
    c, *_ = _check(M, cfg2, -1)
    d, *_ = _check(M, cfg2, 128)
    e, *_ = _check(M, cfg2, 0)
    assert torch.equal(c, d) and torch.equal(d, e)


def test_f8_widths_differ(M):
    cfg = CFGS["many"]
    a, *_ = _check(M, cfg, 64)
    b, *_ = _check(M, cfg, 128)
    assert not torch.equal(a, b)


@pytest.mark.parametrize("gran", [64, 128])
def test_f8_fast_requant_division_is_exact(M, gran):
    """debug_flags bit 4 divides for every requant code; the default divides only
    next to an e4m3 rounding boundary.  Codes, scales and outputs are identical."""
    cfg = CFGS["wide"].with_(seed=64)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    res = []
    for flags in (0, 16):
        opt = M.options(M.MM_MOE_VARIANT_F8, f8_act_gran=gran, debug_flags=flags, retain_intermediate=1)
        out, ws, _, (code, _) = run_forward(M, cfg, dev, opt)
        assert code == 0
        rows = int(M.mm_moe_workspace_region(ws.data_ptr(), opt, cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, 4)[1] // 4)
        codes = torch.empty(rows, cfg.I, dtype=torch.uint8, device="cuda")
        sf = torch.empty(rows, cfg.I // gran, dtype=torch.float32, device="cuda")
        assert M.mm_moe_read_intermediate(ws.data_ptr(), opt, cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, rows,
                                          codes.data_ptr(), sf.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        _, _, slot, _, _ = read_routing(M, cfg, ws, opt)
        live = slot[slot >= 0]
        res.append((out.clone(), codes[live].clone(), sf[live].clone()))
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)


def test_f8_per64_fullsize_sampled_rows(M):
    """The FP8 benchmark shape (T=8192, H=4096, I=2048, E=256, top-8) with per-64
    scales pinned, on the oracle's 1/64 row sample."""
    cfg = W.CONFIGS["f8"]
    dev = W.make_inputs(cfg, "cuda")
    opt = M.options(M.MM_MOE_VARIANT_F8, f8_act_gran=64)
    out, ws, _, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, where
    _, _, slot, _, _ = read_routing(M, cfg, ws, opt)
    rows = W.eval_rows(cfg)
    ref, inter = oracle_rows(cfg, dev, rows, f8_gran=64)
    check_output(out.float().cpu().numpy()[rows], ref, "f8 per-64 full size")
    frac = intermediate_match(M, cfg, ws, opt, slot, inter, "f8 per-64 full size")
    assert frac >= 0.9999, frac
