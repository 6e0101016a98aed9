"""The intermediate as a wrapping ring of R pool blocks in the fused MX stream
(Options.ring_blocks; DeepGEMM PR #440 "Ring sizing, recycling, and why that
granularity"): block b uses slot b % R, a block's L1 tiles wait until the L2
tiles of block b - R have read the slot, and the kernel shortens the lag so that
every such wait points at earlier tiles.  The outputs must be bit-identical to
the whole-pool run (same arithmetic in the same order) and agree with the
oracle; the smallest ring (ceil(T / 128) blocks, which forces lag 0 on skewed
routing), short and long lags, Zipf routing, shared experts, bf16 partials, the
early combine and the flash workload at full size are covered, as are the
timeout path and a routing one expert of which overflows the ring."""
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


def _pair(M, cfg, dev, ring, lag=-1, **kw):
    """(ring run, whole-pool run) with the same options otherwise."""
    opt = lambda r: M.options(M.MM_MOE_VARIANT_MX, fused=1, lag_units=lag, ring_blocks=r, **kw)
    a, _, prep, sa = run_forward(M, cfg, dev, opt(ring))
    assert sa[0] == 0, sa
    a = a.clone()
    b, _, _, sb = run_forward(M, cfg, dev, opt(0), prepared=prep)
    assert sb[0] == 0, sb
    return a, b


def _min_ring(cfg):
    return (cfg.T + 127) // 128


CASES = [
    # name, config, ring (None = the smallest allowed), lag, extra options
    ("ragged-min", W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), None, -1, {}),
    ("ragged-lag0", W.Config("ragged", T=300, H=512, I=384, E=5, K=2, seed=21), 4, 0, {}),
    ("many-experts", W.Config("me", T=256, H=256, I=256, E=64, K=6, seed=61), 5, -1, {}),
    ("many-experts-lag3", W.Config("me", T=256, H=256, I=256, E=64, K=6, seed=61), 6, 3, {}),
    ("zipf-min", W.Config("zipf", T=512, H=256, I=384, E=32, K=4, routing="zipf", seed=62), None, -1, {}),
    ("zipf-wide", W.Config("zipf", T=512, H=256, I=384, E=32, K=4, routing="zipf", seed=62), 9, 8, {}),
    ("early-combine", W.Config("me", T=256, H=256, I=256, E=64, K=6, seed=61), 5, -1, {"early_combine": 1}),
    ("bf16-partials", W.Config("me", T=256, H=256, I=256, E=64, K=6, seed=61), 5, 2, {"partials_bf16": 1}),
    ("shared", W.Config("shared", T=200, H=256, I=256, E=16, K=4, S=1, seed=63), None, -1, {}),
]


@pytest.mark.parametrize("name,cfg,ring,lag,kw", CASES, ids=[c[0] for c in CASES])
def test_ring_bits_equal_whole_pool(M, name, cfg, ring, lag, kw):
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    R = ring if ring is not None else _min_ring(cfg)
    a, b = _pair(M, cfg, dev, R, lag, **kw)
    assert torch.equal(a, b), name
    ref, _ = oracle_rows(cfg, dev, np.arange(cfg.T), keep_intermediate=False,
                         partials_bf16=bool(kw.get("partials_bf16")))
    check_output(a.float().cpu().numpy(), ref, f"{name} ring {R}")


def test_ring_flash_full_size(M):
    """Flash (T=2048, E=256, top-6) with a 64-block ring at lag 29 (PR #440's
    lag rule in experts): bit-identical to the whole pool at the default lag."""
    cfg = W.CONFIGS["flash"]
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    opt = lambda r, lag: M.options(M.MM_MOE_VARIANT_MX, fused=1, lag_units=lag, ring_blocks=r)
    a, _, prep, sa = run_forward(M, cfg, dev, opt(64, 29))
    assert sa[0] == 0, sa
    a = a.clone()
    b, _, _, sb = run_forward(M, cfg, dev, opt(0, -1), prepared=prep)
    assert sb[0] == 0, sb
    assert torch.equal(a, b)


def test_ring_timeout_path(M):
    """debug_flags bit 2 (every L2 tile waits for one more L1 completion than
    arrives) with a ring: the call ends with MM_MOE_ERR_TIMEOUT, nothing hangs,
    and the next call on the same workspace is clean."""
    cfg = W.Config("me", T=256, H=256, I=256, E=64, K=6, seed=61)
    dev = to_dev(W.make_inputs(cfg, "cpu"))
    bad = M.options(M.MM_MOE_VARIANT_MX, fused=1, ring_blocks=3, debug_flags=4, wait_timeout_ms=100)
    out, ws, prep, st = run_forward(M, cfg, dev, bad)
    assert st[0] == M.MM_MOE_ERR_TIMEOUT, st
    good = M.options(M.MM_MOE_VARIANT_MX, fused=1, ring_blocks=3)
    a, _, _, st2 = run_forward(M, cfg, dev, good, prepared=prep)
    assert st2[0] == 0, st2
    b, _, _, st3 = run_forward(M, cfg, dev, M.options(M.MM_MOE_VARIANT_MX, fused=1), prepared=prep)
    assert st3[0] == 0 and torch.equal(a, b)


def test_ring_overfull_expert_is_rejected(M):
    """A routing that names expert 0 in both slots of every token gives it
    2 * ceil(T / 128) blocks, more than the smallest ring holds: the kernel
    reports MM_MOE_ERR_BAD_ROUTING at site 114 instead of waiting."""
    cfg = W.Config("dup", T=200, H=256, I=256, E=8, K=2, seed=64)
    inp = W.make_inputs(cfg, "cpu")
    inp["topk_idx"][:] = 0
    dev = to_dev(inp)
    opt = M.options(M.MM_MOE_VARIANT_MX, fused=1, ring_blocks=_min_ring(cfg), wait_timeout_ms=200)
    _, _, prep, st = run_forward(M, cfg, dev, opt)
    assert st[0] == M.MM_MOE_ERR_BAD_ROUTING and st[1] == 114, st
    _, _, _, st2 = run_forward(M, cfg, dev, M.options(M.MM_MOE_VARIANT_MX, fused=1), prepared=prep)
    assert st2[0] == 0, st2
