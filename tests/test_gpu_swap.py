"""The swapped-operand MX kernels (weights as the MMA's M side, each pool
block's tokens as N rounded up to 16; swap_ab = 1 on single CTAs, swap_ab = 2
on 2-CTA clusters with cta_group::2 MMAs) against the oracle: small and
ragged shapes in both block sizes (80 and 160 tokens) and both launch modes,
masked and out-of-range slots, blocks of more than 128 tokens (two scale
chunks), the largest expert count and top-k, the L1 accumulators themselves,
the early combine, and the numeric options."""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from gpu_util import (check_output, intermediate_match, oracle_rows, read_routing, run_forward, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[1, 2], ids=["single", "pair"])
def sw(request):
    return request.param


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


CFGS = {
    "tiny": W.CONFIGS["tiny"],
    # several blocks per expert at both block sizes, ragged tails, 3 L1 tiles
    "ragged": W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21),
    # H % 256 == 128: the last L2 tile's second half lies past H
    "k1": W.Config("k1", T=77, H=384, I=256, E=3, K=1, seed=22),
    "manyexp": W.Config("manyexp", T=40, H=256, I=128, E=64, K=6, seed=23),
    # 150 tokens per expert: one 160-token block holding two scale chunks
    "wide": W.Config("wide", T=150, H=256, I=256, E=2, K=2, seed=27),
}


def _opt(M, bm, fused, sw, **kw):
    return M.options(M.MM_MOE_VARIANT_MX, swap_ab=sw, block_m=bm, fused=fused, **kw)


def _check(M, cfg, inp, opt, label):
    dev = to_dev(inp)
    out, ws, prepared, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, f"{label}: device status {code} at site {where}"
    cnt, blk, slot, src, bm = read_routing(M, cfg, ws, opt)
    assert bm == opt.block_m
    ref_route = O.route(inp["topk_idx"].numpy(), cfg.E, bm)
    assert np.array_equal(cnt, ref_route["cnt"]) and np.array_equal(blk, ref_route["blk_off"])
    assert np.array_equal(slot, ref_route["slot"])
    assert np.array_equal(src[:len(ref_route["src"])], ref_route["src"])
    ref, inter = oracle_rows(cfg, dev, np.arange(cfg.T))
    check_output(out.float().cpu().numpy(), ref, label)
    frac = intermediate_match(M, cfg, ws, opt, slot, inter, label=label)
    assert frac >= 0.999, f"{label}: intermediate code match {frac:.5f}"
    return out, ws, prepared


@pytest.mark.parametrize("fused", [1, 0])
@pytest.mark.parametrize("bm", [80, 160])
@pytest.mark.parametrize("name", list(CFGS))
def test_swap_parity(M, name, bm, fused, sw):
    cfg = CFGS[name]
    _check(M, cfg, W.make_inputs(cfg, "cpu"), _opt(M, bm, fused, sw), f"swap{sw} {name} bm{bm} fused{fused}")


@pytest.mark.parametrize("bm", [80, 160])
def test_swap_fused_equals_two_launch_bitwise(M, bm, sw):
    """Both launch modes run the same tiles in the same order of k-blocks per block."""
    cfg = CFGS["ragged"].with_(seed=44)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    a, _, prep, sa = run_forward(M, cfg, dev, _opt(M, bm, 0, sw))
    a = a.clone()
    for lag in (0, 2, -1):
        b, _, _, sb = run_forward(M, cfg, dev, _opt(M, bm, 1, sw, lag_units=lag), prepared=prep)
        assert sa[0] == 0 and sb[0] == 0
        assert torch.equal(a, b), lag


@pytest.mark.parametrize("bm", [80, 160])
def test_swap_masked_and_flagged_slots(M, bm, sw):
    cfg = CFGS["ragged"].with_(seed=31)
    inp = W.make_inputs(cfg, "cpu")
    g = torch.Generator().manual_seed(5)
    inp["topk_idx"][torch.rand(cfg.T, cfg.K, generator=g) < 0.2] = -1
    inp["topk_idx"][7, :] = -1
    out, _, _ = _check(M, cfg, inp, _opt(M, bm, 1, sw), f"swap masked bm{bm}")
    assert torch.all(out[7] == 0)
    bad = {k: v.clone() for k, v in inp.items()}
    bad["topk_idx"][9, 1] = -2
    bad["topk_idx"][11, 0] = cfg.E + 5
    dev = to_dev(bad)
    got, _, _, (code, _) = run_forward(M, cfg, dev, _opt(M, bm, 1, sw))
    assert code == M.MM_MOE_ERR_BAD_ROUTING
    ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False)
    check_output(got.float().cpu().numpy(), ref, "swap flagged slots")


@pytest.mark.parametrize("name,cfg", [
    ("e1024", W.Config("e1024", T=96, H=256, I=128, E=1024, K=4, seed=34)),
    ("k16", W.Config("k16", T=40, H=256, I=256, E=32, K=16, seed=35)),
    ("t1", W.Config("t1", T=1, H=128, I=128, E=1, K=1, seed=36)),
    ("skew", W.Config("skew", T=700, H=256, I=128, E=3, K=1, seed=37)),   # ~233 tokens/expert: 2-3 blocks each
])
def test_swap_edges(M, name, cfg, sw):
    for bm in (80, 160):
        _check(M, cfg, W.make_inputs(cfg, "cpu"), _opt(M, bm, 1, sw), f"swap{sw} {name} bm{bm}")


@pytest.mark.parametrize("bm", [80, 160])
def test_swap_l1_accumulators_match_oracle(M, bm, sw):
    """Debug mode: the raw fp32 gate|up sums against the oracle's fp64 gate|up."""
    cfg = CFGS["ragged"]
    inp = W.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    opt = _opt(M, bm, 0, sw, debug_flags=1)
    out, ws, _, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, where
    dbg = M.workspace_view(ws, opt, cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, "debug", torch.float32)
    dbg = dbg.view(-1, 2 * cfg.I).cpu().numpy().astype(np.float64)
    _, _, slot, _, _ = read_routing(M, cfg, ws, opt)
    npi = {k: v.numpy() for k, v in inp.items()}
    errs = []
    for t in range(0, cfg.T, 7):
        xh = O.dequant_x(npi["x"][t], npi["x_sf"][t], "mx")
        for k in range(cfg.K):
            e = int(npi["topk_idx"][t, k])
            W1 = O.dequant_weight(npi["w1"][e], npi["w1_sf"][e], "mx")
            ref = W1 @ xh
            errs.append(np.max(np.abs(dbg[slot[t, k]] - ref)) / (np.max(np.abs(ref)) + 1e-30))
    assert max(errs) < 1e-5, max(errs)


@pytest.mark.parametrize("kw", [dict(early_combine=1), dict(partials_bf16=1), dict(activation_clamp=0.05),
                                dict(precise_swiglu=1), dict(partials_bf16=1, early_combine=1)],
                         ids=["early-combine", "bf16-partials", "clamp", "precise", "bf16-early"])
def test_swap_options(M, kw, sw):
    cfg = CFGS["ragged"].with_(seed=45)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    for bm in (80, 160):
        opt = _opt(M, bm, 1, sw, **kw)
        out, ws, _, (code, where) = run_forward(M, cfg, dev, opt)
        assert code == 0, (kw, where)
        ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False,
                             partials_bf16=bool(kw.get("partials_bf16")),
                             clamp=kw.get("activation_clamp"))
        check_output(out.float().cpu().numpy(), ref, f"swap {kw} bm{bm}")
    if kw.get("early_combine"):   # the early combine gives the combine kernel's bits
        base = dict(kw, early_combine=0)
        a, _, prep, _ = run_forward(M, cfg, dev, _opt(M, 160, 1, sw, **kw))
        a = a.clone()
        b, _, _, _ = run_forward(M, cfg, dev, _opt(M, 160, 1, sw, **base), prepared=prep)
        assert torch.equal(a, b)


def test_swap_x_bf16_matches_prequantised(M, sw):
    """bf16 activations quantised in the gather give the bits of feeding the
    oracle's own quantisation of the same rows."""
    cfg = CFGS["ragged"].with_(seed=46)
    inp = W.make_inputs(cfg, "cpu")
    xb = W.make_x_bf16(cfg, "cpu")
    q, qsf = O.quantise_x(xb.float().numpy(), "mx")
    dq = to_dev(dict(inp, x=torch.from_numpy(q), x_sf=torch.from_numpy(np.ascontiguousarray(qsf))))
    for fused in (1, 0):
        a, _, prep, sa = run_forward(M, cfg, dq, _opt(M, 160, fused, sw))
        a = a.clone()
        db = dict(dq, x=xb.cuda(), x_sf=None)
        b, _, _, sb = run_forward(M, cfg, db, _opt(M, 160, fused, sw, x_bf16=1), prepared=prep)
        assert sa[0] == 0 and sb[0] == 0
        assert torch.equal(a, b), fused


def test_swap_rejects_unsupported_blocks(M):
    cfg = CFGS["tiny"]
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    for bad in (dict(swap_ab=1, block_m=128), dict(swap_ab=2, block_m=96), dict(swap_ab=0, block_m=80),
                dict(swap_ab=2, block_m=128)):
        with pytest.raises(M.MMError) as ei:
            run_forward(M, cfg, dev, M.options(**bad))
        assert ei.value.code == M.MM_MOE_ERR_UNSUPPORTED, bad
