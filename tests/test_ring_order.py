"""Why the intermediate ring cannot deadlock, checked on the CPU.

The fused stream deals tile groups in segments: segment u holds expert u's L1
groups, then expert (u - lag)'s L2 groups (DeepGEMM PR #440 "How it works").
With a ring of R pool blocks, block b's L1 tiles wait until the L2 tiles of block
b - R have read the slot, so every L2 group that reads block b - R must come
before every L1 group that writes block b.  The kernel picks the lag from the
block offsets: the largest lag <= the requested one whose windows of lag + 1
consecutive experts own at most R / 2 blocks, or 0 when one expert alone owns
more than R / 2 (and it refuses a routing where one expert owns more than R).
This test restates that rule and the group order and checks the property, plus
the slack, on random routings of both distributions."""
import numpy as np
import pytest


def _blocks(cnt, bt=128):
    return [(c + bt - 1) // bt for c in cnt]


def _window_max(nb, lag):
    off = np.concatenate([[0], np.cumsum(nb)])
    E = len(nb)
    return max(off[u + 1] - off[max(0, u - lag)] for u in range(E))


def _ring_lag(nb, lag, R):
    """The rule the kernel applies at launch."""
    if _window_max(nb, 0) > R:
        return None                                 # refused: BAD_ROUTING
    half = R // 2
    if _window_max(nb, 0) > half:
        return 0
    best = 0
    for l in range(lag + 1):                        # windows grow with the lag
        if _window_max(nb, l) <= half:
            best = l
    return best


def _stream(nb, lag, NB1=2, NB2=2):
    """Group index of every (type, expert, tile) in the lag-ordered stream."""
    E = len(nb)
    order = {}
    g = 0
    for u in range(E + lag):
        if u < E and nb[u]:
            for n in range(NB1):
                order[(1, u, n)] = g
                g += 1
        v = u - lag
        if 0 <= v < E and nb[v]:
            for n in range(NB2):
                order[(2, v, n)] = g
                g += 1
    return order


def _check(cnt, lag, R):
    nb = _blocks(cnt)
    lg = _ring_lag(nb, lag, R)
    if lg is None:
        assert _window_max(nb, 0) > R
        return None
    assert lg <= lag
    order = _stream(nb, lg)
    owner = np.repeat(np.arange(len(nb)), nb)       # expert of each pool block
    for b in range(R, len(owner)):
        e_new, e_old = owner[b], owner[b - R]
        last_reader = max(order[(2, e_old, n)] for n in range(2))
        first_writer = min(order[(1, e_new, n)] for n in range(2))
        assert last_reader < first_writer, (b, e_new, e_old, lg)
    if _window_max(nb, 0) <= R // 2:
        assert _window_max(nb, lg) <= R // 2        # half the ring stays slack
    return lg


def _routing(rng, T, K, E, zipf):
    if zipf:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        logits = np.log(p)[rng.permutation(E)]
    else:
        logits = np.zeros(E)
    keys = logits[None, :] + rng.gumbel(size=(T, E))
    idx = np.argsort(-keys, axis=1)[:, :K]
    return np.bincount(idx.ravel(), minlength=E)


@pytest.mark.parametrize("zipf", [False, True])
def test_ring_waits_point_at_earlier_groups(zipf):
    rng = np.random.default_rng(7 + zipf)
    checked = 0
    for _ in range(300):
        E = int(rng.integers(1, 48))
        K = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.integers(1, 1500))
        lag = int(rng.integers(0, E + 1))
        R = int(rng.integers((T + 127) // 128, (T + 127) // 128 + 40))
        cnt = _routing(rng, T, K, E, zipf)
        if _check(cnt, lag, R) is not None:
            checked += 1
    assert checked == 300                           # distinct experts per token: never refused


def test_the_full_lag_would_break_the_order_without_the_rule():
    """Counter-check: with a ring smaller than a window, keeping the requested lag
    puts an L2 reader after the L1 writer it must precede."""
    cnt = [128] * 8                                 # one block per expert
    nb = _blocks(cnt)
    R, lag = 3, 7
    order = _stream(nb, lag)
    bad = any(order[(2, b - R, 0)] > order[(1, b, 0)] for b in range(R, 8))
    assert bad
    assert _ring_lag(nb, lag, R) == 0 and _check(cnt, lag, R) == 0


def test_an_expert_named_twice_overflows_the_smallest_ring():
    cnt = [400, 0, 0]                               # T = 200, K = 2, both slots on expert 0
    assert _check(cnt, 2, 2) is None


def test_every_l2_group_follows_its_blocks_l1_groups():
    """The stream's own dependency (an L2 tile reads blocks the expert's L1 tiles
    wrote) points backwards for every lag, ring or not."""
    rng = np.random.default_rng(11)
    for _ in range(100):
        E = int(rng.integers(1, 40))
        nb = list(rng.integers(0, 4, size=E))
        for lag in (0, 1, int(rng.integers(0, E + 1)), E):
            order = _stream(nb, lag)
            for v in range(E):
                if nb[v]:
                    assert max(order[(1, v, n)] for n in range(2)) < min(order[(2, v, n)] for n in range(2))
