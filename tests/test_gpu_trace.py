"""The per-task trace of the token-M MX kernel (Options.trace_buf): every task
of the stream appears exactly once, with its CTA's task indices in order and
its timestamps ordered, in the fused stream and in both launches of the
two-launch path; tracing changes no output bit; a buffer below one record per
CTA and launch, and the F8 variant, are refused."""
import numpy as np
import pytest
import torch

import workload as W
from gpu_util import read_routing, run_forward, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


def _expected(cfg, cnt, blk):
    NB1, NB2 = cfg.I // 128, (cfg.H + 255) // 256
    want = []
    for e in range(cfg.E):
        nb = blk[e + 1] - blk[e]
        for b in range(blk[e], blk[e] + nb):
            want += [(1, e, n, b) for n in range(NB1)] + [(2, e, n, b) for n in range(NB2)]
    return sorted(want)


@pytest.mark.parametrize("fused", [1, 0])
def test_trace_lists_every_task_once(M, fused):
    from moe_expert_forward_gb300 import trace as TR
    cfg = W.Config("tr", T=300, H=512, I=384, E=12, K=3, seed=95)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    plain, _, prep, st = run_forward(M, cfg, dev, M.options(M.MM_MOE_VARIANT_MX, fused=fused))
    assert st[0] == 0
    plain = plain.clone()
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(TR.buffer_bytes(grid, 64, 1 if fused else 2), dtype=torch.uint8, device="cuda")
    opt = M.options(M.MM_MOE_VARIANT_MX, fused=fused, trace_buf=buf.data_ptr(), trace_bytes=buf.numel())
    out, ws, _, st = run_forward(M, cfg, dev, opt, prepared=prep)
    assert st[0] == 0 and torch.equal(out, plain)
    cnt, blk, _, _, _ = read_routing(M, cfg, ws, opt)
    rec = TR.records(buf)
    got = sorted((int(r["type"]), int(r["expert"]), int(r["tile"]), int(r["block"])) for r in rec)
    assert got == _expected(cfg, cnt, blk)
    assert set(np.unique(rec["mode"])) == ({3} if fused else {1, 2})
    for mode in np.unique(rec["mode"]):
        for c in np.unique(rec["cta"]):
            r = rec[(rec["cta"] == c) & (rec["mode"] == mode)]
            assert list(r["task"]) == list(range(r.size))               # in the CTA's order, none lost
    assert (rec["t_issue"] > 0).all()
    assert (rec["t_issue"] <= rec["t_mma_done"]).all() and (rec["t_mma_done"] <= rec["t_epi_done"]).all()
    s = TR.summary(rec)
    assert sum(v["tasks"] for v in s.values()) == rec.size


def test_trace_refusals(M):
    cfg = W.Config("tr", T=64, H=256, I=128, E=8, K=2, seed=96)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")              # one record: fewer than one per CTA
    with pytest.raises(M.MMError) as ei:
        run_forward(M, cfg, dev, M.options(M.MM_MOE_VARIANT_MX, trace_buf=buf.data_ptr(), trace_bytes=64))
    assert ei.value.code == M.MM_MOE_ERR_INVALID_ARG
    f8 = W.Config("tr8", T=64, H=256, I=128, E=8, K=2, variant="f8", seed=97)
    dev8 = to_dev(W.make_inputs(f8, "cpu"))
    big = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MMError) as ei:
        run_forward(M, f8, dev8, M.options(M.MM_MOE_VARIANT_F8, trace_buf=big.data_ptr(), trace_bytes=1 << 20))
    assert ei.value.code == M.MM_MOE_ERR_UNSUPPORTED
