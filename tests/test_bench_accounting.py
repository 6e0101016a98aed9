"""bench.py's byte and FLOP accounting (the denominators of every roofline
fraction it reports) against the figures derived independently from the method's
definition: algorithmic bytes = the weights + scales of every touched expert
(MX: 3·I·H·(1/2 + 1/32) bytes; F8: 3·I·H + the 128×128 fp32 scales), x and its
scales, topk_idx + topk_w and the bf16 output; FLOPs = 6·T·K·H·I over the routed
pairs.  With every expert touched (uniform routing at these sizes touches all of
them), the flash, pro and FP8 workloads come to 3.448, 13.655 and 6.546 GB and
6.18e11, 6.49e12 and 3.30e12 FLOPs."""
import numpy as np
import pytest

import workload as W


def _all_touched(cfg):
    t = np.arange(cfg.T)[:, None]
    k = np.arange(cfg.K)[None, :]
    return ((t * cfg.K + k) % cfg.E).astype(np.int32)     # every expert, K distinct per token when K <= E


@pytest.mark.parametrize("name,gb,flops", [("flash", 3.448, 6.18e11), ("pro", 13.655, 6.49e12),
                                           ("f8", 6.546, 3.30e12)])
def test_step_bytes_and_flops(name, gb, flops):
    import bench
    cfg = W.CONFIGS[name]
    acc = bench.workload_accounting(cfg, _all_touched(cfg))
    assert acc["touched_experts"] == cfg.E and acc["pairs"] == cfg.T * cfg.K
    assert round(acc["step_bytes"] / 1e9, 3) == gb
    assert acc["flops"] == pytest.approx(flops, rel=5e-3)
    assert acc["l1_flops"] + acc["l2_flops"] == acc["flops"]


def test_masked_and_shared_slots_count_as_the_method_counts_them():
    import bench
    cfg = W.Config("acc", T=64, H=256, I=128, E=8, K=2, seed=0)
    idx = _all_touched(cfg)
    idx[::2, 1] = -1                                       # masked slots carry no pair
    acc = bench.workload_accounting(cfg, idx)
    assert acc["pairs"] == cfg.T * cfg.K - cfg.T // 2
    shared = bench.workload_accounting(cfg.with_(S=1), idx)
    assert acc["touched_experts"] == 6                     # experts 1 and 5 were only ever in masked slots
    assert shared["touched_experts"] == acc["touched_experts"] + 1 and shared["pairs"] == acc["pairs"] + cfg.T
    w = 3 * cfg.I * cfg.H * (0.5 + 1 / 32)                 # one more expert's weights and scales
    assert shared["step_bytes"] - acc["step_bytes"] == pytest.approx(w)
