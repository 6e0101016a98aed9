"""End-to-end parity of the forward (MX format) against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from gpu_util import (check_output, intermediate_match, oracle_rows, read_routing, run_forward, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


SMALL = {
    "tiny": W.CONFIGS["tiny"],
    # several token blocks per expert, ragged tails (not multiples of 16/32), 3 L1 weight tiles per 128 rows
    "ragged": W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21),
    "k1": W.Config("k1", T=77, H=384, I=256, E=3, K=1, seed=22),
    "manyexp": W.Config("manyexp", T=40, H=256, I=128, E=64, K=6, seed=23),
    # FP8 x FP8 with fp32 per-128 scales
    "f8_tiny": W.Config("f8_tiny", T=24, H=256, I=256, E=4, K=2, variant="f8", seed=24),
    "f8_ragged": W.Config("f8_ragged", T=300, H=512, I=384, E=5, K=2, variant="f8", seed=25),
    "f8_wide": W.Config("f8_wide", T=150, H=384, I=512, E=3, K=3, variant="f8", seed=26),
}


def _opt_for(M, cfg, **kw):
    return M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8, **kw)


def _full_check(M, cfg, inp, opt=None):
    opt = opt or _opt_for(M, cfg)
    dev = to_dev(inp)
    out, ws, prepared, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, f"device status {code} at site {where}"
    cnt, blk, slot, src, bm = read_routing(M, cfg, ws, opt)
    ref_route = O.route(inp["topk_idx"].numpy(), cfg.E, bm)
    assert np.array_equal(cnt, ref_route["cnt"]) and np.array_equal(blk, ref_route["blk_off"])
    assert np.array_equal(slot, ref_route["slot"])
    assert np.array_equal(src[:len(ref_route["src"])], ref_route["src"])
    rows = np.arange(cfg.T)
    ref, inter = oracle_rows(cfg, dev, rows)
    got = out.float().cpu().numpy()
    stats = check_output(got, ref, cfg.name)
    frac = intermediate_match(M, cfg, ws, opt, slot, inter)
    assert frac >= 0.999, f"intermediate code match {frac:.5f}"
    return out, stats


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small_configs(M, name):
    cfg = SMALL[name]
    _full_check(M, cfg, W.make_inputs(cfg, "cpu"))


def test_forward_masked_slots(M):
    cfg = SMALL["ragged"].with_(seed=31)
    inp = W.make_inputs(cfg, "cpu")
    g = torch.Generator().manual_seed(5)
    mask = torch.rand(cfg.T, cfg.K, generator=g) < 0.2
    inp["topk_idx"][mask] = -1
    inp["topk_idx"][7, :] = -1                       # a token with no expert at all
    out, _ = _full_check(M, cfg, inp)
    assert torch.all(out[7] == 0)


def test_forward_repeatable_and_grid_independent(M):
    cfg = SMALL["ragged"].with_(seed=41)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    out1, ws, prep, st = run_forward(M, cfg, dev)
    out1 = out1.clone()
    out2, _, _, _ = run_forward(M, cfg, dev, ws=ws, prepared=prep)
    assert torch.equal(out1, out2)
    out3, _, _, st3 = run_forward(M, cfg, dev, opt=M.options(num_sms=7), prepared=prep)
    assert st3[0] == 0 and torch.equal(out1, out3)


def test_forward_zero_weights_gives_zero(M):
    cfg = SMALL["tiny"].with_(seed=51)
    inp = W.make_inputs(cfg, "cpu")
    inp["w2"].zero_()
    dev = to_dev(inp)
    out, ws, _, (code, _) = run_forward(M, cfg, dev)
    assert code == 0 and torch.all(out == 0)


def test_forward_l1_accumulators_match_oracle(M):
    """Debug mode: the raw fp32 gate|up accumulators of the L1 GEMM against the
    oracle's fp64 gate|up for every routed pair."""
    cfg = SMALL["ragged"]
    inp = W.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    opt = M.options(debug_flags=1)
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
            got = dbg[slot[t, k]]
            errs.append(np.max(np.abs(got - ref)) / (np.max(np.abs(ref)) + 1e-30))
    assert max(errs) < 1e-5, max(errs)


@pytest.mark.parametrize("lag", [0, 1, 3, 64, -1])
@pytest.mark.parametrize("name", ["tiny", "ragged", "manyexp", "k1"])
def test_fused_stream_bitwise_equals_two_launch_path(M, name, lag):
    """The lag-ordered single-launch stream computes every tile exactly as the
    two-launch path does, whatever the lag: outputs and intermediates are equal bit for bit."""
    cfg = SMALL[name]
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    out_a, ws_a, prep, st_a = run_forward(M, cfg, dev, M.options(fused=0))
    out_a = out_a.clone()
    out_b, ws_b, _, st_b = run_forward(M, cfg, dev, M.options(fused=1, lag_units=lag), prepared=prep)
    assert st_a[0] == 0 and st_b[0] == 0, (st_a, st_b)
    assert torch.equal(out_a, out_b)
    opt = M.options()
    pa = M.workspace_view(ws_a, opt, cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, "pool2")
    pb = M.workspace_view(ws_b, opt, cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, "pool2")
    _, blk, _, src, _ = read_routing(M, cfg, ws_a, opt)
    live = torch.from_numpy(src[:blk[-1] * 128] >= 0)
    rows = pa.view(-1, cfg.I)[:blk[-1] * 128][live.cuda()]
    assert torch.equal(rows, pb.view(-1, cfg.I)[:blk[-1] * 128][live.cuda()])


@pytest.mark.parametrize("pairs", [2, 3, -1])
def test_reserved_cta_pairs_values_are_rejected(M, pairs):
    """cta_pairs is reserved: only 0 and 1 are accepted, before any launch."""
    cfg = SMALL["tiny"]
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    with pytest.raises(M.MMError) as ei:
        run_forward(M, cfg, dev, M.options(cta_pairs=pairs))
    assert ei.value.code == M.MM_MOE_ERR_UNSUPPORTED
    out, _, _, (code, _) = run_forward(M, cfg, dev, M.options(cta_pairs=1))
    assert code == 0


def test_fused_stream_parity_and_masking(M):
    cfg = SMALL["ragged"].with_(seed=61)
    inp = W.make_inputs(cfg, "cpu")
    g = torch.Generator().manual_seed(7)
    inp["topk_idx"][torch.rand(cfg.T, cfg.K, generator=g) < 0.15] = -1
    _full_check(M, cfg, inp, M.options(fused=1))


@pytest.mark.parametrize("variant", ["mx", "f8"])
def test_timing_events_do_not_change_the_result(M, variant):
    """With events between its kernels the library launches them plainly, without
    them programmatically (the GEMM and the combine start early and wait
    in-kernel); NULL entries are skipped.  All three give the same bits."""
    import ctypes
    cfg = W.Config("ev", T=200, H=512, I=256, E=6, K=3, variant=variant, seed=61)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    var = M.MM_MOE_VARIANT_MX if variant == "mx" else M.MM_MOE_VARIANT_F8
    a, _, prep, sa = run_forward(M, cfg, dev, M.options(var))
    a = a.clone()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(M.MM_MOE_NUM_TIMING_EVENTS)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    outs = []
    for handles in ([e.cuda_event for e in evs], [evs[0].cuda_event] + [None] * 4 + [evs[-1].cuda_event]):
        arr = (ctypes.c_void_p * M.MM_MOE_NUM_TIMING_EVENTS)(*handles)
        o = M.options(var)
        o.timing_events = ctypes.cast(arr, ctypes.c_void_p)
        b, _, _, sb = run_forward(M, cfg, dev, o, prepared=prep)
        torch.cuda.synchronize()
        assert sb[0] == 0, sb
        outs.append(b.clone())
    assert sa[0] == 0
    assert all(torch.equal(a, b) for b in outs)
