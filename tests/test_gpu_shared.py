"""Shared experts (Options.shared_experts): experts E .. E+S-1 that every token
uses with weight 1 after its routed slots, computed in the same launches as the
routed experts, against the oracle (shared=S); the routing they add is checked
bit for bit against the oracle's routing of the extended table."""
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


CFGS = {
    "mx_s1": W.Config("sh_mx_s1", T=300, H=512, I=384, E=5, K=2, seed=71, S=1),
    "mx_s2": W.Config("sh_mx_s2", T=130, H=256, I=256, E=16, K=4, seed=72, S=2),
    "f8_s1": W.Config("sh_f8_s1", T=200, H=512, I=256, E=6, K=2, variant="f8", seed=73, S=1),
}


def _opt(M, cfg, **kw):
    return M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8, **kw)


def _extended(idx: np.ndarray, E: int, S: int) -> np.ndarray:
    """The routing table with the S shared slots appended (what the library routes)."""
    T = idx.shape[0]
    ext = np.where((idx >= E) & (idx < E + S), -2, idx)
    return np.concatenate([ext, np.tile(np.arange(E, E + S, dtype=idx.dtype), (T, 1))], 1)


def _check(M, cfg, opt, inp=None, status=0):
    inp = inp if inp is not None else W.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    out, ws, _, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == status, f"device status {code} at site {where}"
    cnt, blk, slot, src, bm = read_routing(M, cfg, ws, opt)
    ref_route = O.route(_extended(inp["topk_idx"].numpy(), cfg.E, cfg.S), cfg.E + cfg.S, bm)
    assert np.array_equal(cnt, ref_route["cnt"]) and np.array_equal(blk, ref_route["blk_off"])
    assert np.array_equal(slot, ref_route["slot"])
    assert np.array_equal(src[:len(ref_route["src"])], ref_route["src"])
    ref, inter = oracle_rows(cfg, dev, np.arange(cfg.T))
    check_output(out.float().cpu().numpy(), ref, f"{cfg.name} shared")
    frac = intermediate_match(M, cfg, ws, opt, slot, inter, f"{cfg.name} shared")
    assert frac >= 0.999, frac
    return out.clone()


FORMS = {"fused": dict(), "two_launch": dict(fused=0), "swap": dict(swap_ab=1), "pairs": dict(swap_ab=2),
         "early_combine": dict(early_combine=1)}


@pytest.mark.parametrize("form", list(FORMS))
@pytest.mark.parametrize("name", ["mx_s1", "mx_s2"])
def test_shared_experts_mx_match_oracle(M, name, form):
    cfg = CFGS[name]
    _check(M, cfg, _opt(M, cfg, **FORMS[form]))


def test_shared_experts_f8_match_oracle(M):
    cfg = CFGS["f8_s1"]
    _check(M, cfg, _opt(M, cfg))


def test_shared_experts_fused_equals_two_launch(M):
    cfg = CFGS["mx_s2"]
    a = _check(M, cfg, _opt(M, cfg))
    b = _check(M, cfg, _opt(M, cfg, fused=0))
    assert torch.equal(a, b)


def test_shared_expert_alone(M):
    """Every routed slot masked: the output is the shared expert's MLP on every token."""
    cfg = CFGS["mx_s1"].with_(seed=74)
    inp = W.make_inputs(cfg, "cpu")
    inp["topk_idx"].fill_(-1)
    out = _check(M, cfg, _opt(M, cfg), inp)
    assert torch.all(out.float().abs().amax(1) > 0)


def test_routed_id_naming_a_shared_expert_is_flagged(M):
    """topk_idx names routed experts only: an id in [E, E+S) is out of range, so
    it is masked and the call reports MM_MOE_ERR_BAD_ROUTING."""
    cfg = CFGS["mx_s2"].with_(seed=75)
    inp = W.make_inputs(cfg, "cpu")
    inp["topk_idx"][3, 1] = cfg.E
    inp["topk_idx"][9, 0] = cfg.E + 1
    bad = _check(M, cfg, _opt(M, cfg), inp, status=M.MM_MOE_ERR_BAD_ROUTING)
    masked = {k: v.clone() for k, v in inp.items()}
    masked["topk_idx"][3, 1] = -1
    masked["topk_idx"][9, 0] = -1
    ok = _check(M, cfg, _opt(M, cfg), masked)
    assert torch.equal(bad, ok)


def test_shared_experts_fill_sixteen_slots(M):
    cfg = W.Config("sh_k16", T=40, H=256, I=128, E=24, K=12, seed=76, S=4)
    _check(M, cfg, _opt(M, cfg))


def test_shared_expert_fullsize_flash_sampled_rows(M):
    """The flash shape with one shared expert (2048 more rows, 16 blocks of one
    expert), on the oracle's 1/64 row sample."""
    cfg = W.CONFIGS["flash"].with_(S=1)
    dev = W.make_inputs(cfg, "cuda")
    opt = _opt(M, cfg)
    out, ws, _, (code, where) = run_forward(M, cfg, dev, opt)
    assert code == 0, where
    _, _, slot, _, _ = read_routing(M, cfg, ws, opt)
    rows = W.eval_rows(cfg)
    ref, inter = oracle_rows(cfg, dev, rows)
    check_output(out.float().cpu().numpy()[rows], ref, "flash + 1 shared expert")
    frac = intermediate_match(M, cfg, ws, opt, slot, inter, "flash + 1 shared expert")
    assert frac >= 0.999, frac
