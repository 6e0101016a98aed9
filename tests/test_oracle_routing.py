"""Pins for the oracle's routing (dispatch: histogram, segment offsets, slots)."""
import os

import numpy as np
import pytest

import oracle as O
import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    blocks = []
    cur = None
    with open(os.path.join(GOLDEN, "routing_pool_segments.txt")) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            key, *vals = ln.split()
            vals = [int(v) for v in vals]
            if key == "counts":
                counts = vals
            elif key == "block_m":
                cur = {"block_m": vals[0]}
                blocks.append(cur)
            else:
                cur[key] = vals
    return counts, blocks


@pytest.mark.parametrize("case", range(2))
def test_worked_example_pool_segments(case):
    counts, blocks = _golden()
    g = blocks[case]
    # tokens 0..99 -> e0, 100..109 -> e1, 110..139 -> e2 (K = 1), visited in a shuffled order
    # of experts per token is irrelevant with K = 1; the dense order is by token index.
    idx = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).reshape(-1, 1)
    r = O.route(idx, 3, g["block_m"])
    assert list(r["cnt"]) == counts
    assert list(r["blk_off"]) == g["blk_off"]
    for e in range(3):
        rows = np.sort(r["slot"][idx[:, 0] == e, 0])
        lo, hi = g[f"rows_e{e}"]
        assert list(rows) == list(range(lo, hi + 1))


def _brute(idx, E, block):
    """Sort of (expert, token, slot) triples -> pool rows; independent of route()."""
    T, K = idx.shape
    trip = sorted((int(idx[t, k]), t, k) for t in range(T) for k in range(K) if 0 <= idx[t, k] < E)
    slot = -np.ones((T, K), dtype=np.int64)
    row, prev = 0, None
    for e, t, k in trip:
        if e != prev:
            row = (row + block - 1) // block * block   # start of a new aligned segment
            prev = e
        slot[t, k] = row
        row += 1
    return slot


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("block", [16, 64, 128])
def test_route_matches_brute_force_sort(seed, block):
    rng = np.random.default_rng(seed)
    T, E, K = int(rng.integers(1, 70)), int(rng.integers(1, 12)), 1
    K = int(rng.integers(1, min(E, 4) + 1))
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)])
    idx[rng.random(idx.shape) < 0.1] = -1                     # masked slots
    r = O.route(idx, E, block)
    b = _brute(idx, E, block)
    # experts with no tokens occupy no rows in both; compare slots directly
    assert np.array_equal(r["slot"], b)


@pytest.mark.parametrize("name", ["tiny", "flash", "decode"])
def test_route_invariants_on_workload(name):
    cfg = W.CONFIGS[name]
    idx, _ = W.make_routing(cfg, "cpu")
    idx = idx.numpy()
    block = 128
    r = O.route(idx, cfg.E, block)
    T, K = idx.shape
    assert r["cnt"].sum() == T * K and r["bad"] == 0
    assert all(len(set(row)) == K for row in idx)                   # distinct experts per token
    assert r["blk_off"][-1] == sum((c + block - 1) // block for c in r["cnt"])
    assert np.all(np.diff(r["blk_off"]) >= 0)
    src = r["src"]
    assert np.count_nonzero(src >= 0) == T * K
    tok = src[src >= 0] // K
    assert np.array_equal(np.bincount(tok, minlength=T), np.full(T, K))   # each token K times
    for e in range(cfg.E):
        rows = np.arange(r["blk_off"][e] * block, r["blk_off"][e] * block + r["cnt"][e])
        assert np.all(idx.reshape(-1)[src[rows]] == e)
        assert np.all(np.diff(src[rows] // K) > 0)                  # ascending token index
        pad = np.arange(r["blk_off"][e] * block + r["cnt"][e], r["blk_off"][e + 1] * block)
        assert np.all(src[pad] == -1)


def test_route_masked_and_out_of_range():
    idx = np.array([[0, -1], [5, 1], [1, 0], [-3, 7]])
    r = O.route(idx, 4, 4)
    assert list(r["cnt"]) == [2, 2, 0, 0]
    assert r["bad"] == 3                      # 5 and 7 (>= E), -3 (< -1)
    assert r["slot"][0, 1] == -1 and r["slot"][1, 0] == -1 and r["slot"][3, 1] == -1
    assert r["slot"][0, 0] == 0 and r["slot"][2, 1] == 1 and r["slot"][1, 1] == 4 and r["slot"][2, 0] == 5


def test_zipf_routing_is_skewed():
    cfg = W.CONFIGS["decode"]
    idx, w = W.make_routing(cfg, "cpu")
    cnt = np.bincount(idx.numpy().reshape(-1), minlength=cfg.E)
    assert cnt.max() > 40 and np.count_nonzero(cnt) < cfg.E
    assert np.allclose(w.sum(1).numpy(), 1.0, atol=1e-6)
