"""Step a1 (dispatch) on the GPU against the oracle's routing: bit-exact."""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


def _dispatch(M, idx: np.ndarray, E: int, block: int, scratch_bytes=None):
    T, K = idx.shape
    d_idx = torch.from_numpy(idx.astype(np.int32)).cuda()
    cap = T * K + min(T * K, E) * (block - 1) + 1
    cnt = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    blk = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    slot = torch.full((max(T * K, 1),), -7, dtype=torch.int32, device="cuda")
    src = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    nscr = M.mm_moe_dispatch_scratch_size(T, K, E) if scratch_bytes is None else scratch_bytes
    scratch = torch.empty(max(nscr, 4), dtype=torch.uint8, device="cuda")
    r = M.mm_moe_dispatch(d_idx.data_ptr(), T, K, E, block, cnt.data_ptr(), blk.data_ptr(), slot.data_ptr(),
                          src.data_ptr(), cap, scratch.data_ptr(), nscr, status.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    assert r == 0
    torch.cuda.synchronize()
    return cnt.cpu().numpy(), blk.cpu().numpy(), slot.cpu().numpy()[:T * K].reshape(T, K), src.cpu().numpy(), \
        int(status[0])


@pytest.mark.parametrize("name", ["tiny", "flash", "decode", "pro", "f8"])
def test_dispatch_workload_bit_exact(M, name):
    cfg = W.CONFIGS[name]
    idx, _ = W.make_routing(cfg, "cpu")
    idx = idx.numpy()
    cnt, blk, slot, src, st = _dispatch(M, idx, cfg.E, 128)
    ref = O.route(idx, cfg.E, 128)
    assert st == 0
    assert np.array_equal(cnt, ref["cnt"])
    assert np.array_equal(blk, ref["blk_off"])
    assert np.array_equal(slot, ref["slot"])
    n = len(ref["src"])
    assert np.array_equal(src[:n], ref["src"])
    assert np.all(src[n:] == -7)           # rows past the last block are untouched


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("block", [16, 64, 128, 256])
def test_dispatch_ragged_masked(M, seed, block):
    rng = np.random.default_rng(100 + seed)
    T, E = int(rng.integers(1, 3000)), int(rng.integers(2, 300))
    K = int(rng.integers(1, min(E, 8) + 1))
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[rng.random(idx.shape) < 0.05] = -1
    cnt, blk, slot, src, st = _dispatch(M, idx, E, block)
    ref = O.route(idx, E, block)
    assert st == 0
    assert np.array_equal(cnt, ref["cnt"]) and np.array_equal(blk, ref["blk_off"])
    assert np.array_equal(slot, ref["slot"])
    assert np.array_equal(src[:len(ref["src"])], ref["src"])


@pytest.mark.parametrize("bad", [9, -2])
def test_dispatch_flags_out_of_range_experts(M, bad):
    idx = np.array([[0, 3], [bad, 1], [2, -1]], dtype=np.int32)
    cnt, blk, slot, src, st = _dispatch(M, idx, 4, 16)
    ref = O.route(idx, 4, 16)
    assert st == M.MM_MOE_ERR_BAD_ROUTING
    assert np.array_equal(slot, ref["slot"]) and np.array_equal(cnt, ref["cnt"])


@pytest.mark.parametrize("ctas", [1, 3, 17])
def test_dispatch_fewer_ctas_same_result(M, ctas):
    """A smaller scratch means fewer CTAs; the routing must not change."""
    cfg = W.CONFIGS["flash"]
    idx, _ = W.make_routing(cfg, "cpu")
    idx = idx.numpy()
    full = _dispatch(M, idx, cfg.E, 128)
    part = _dispatch(M, idx, cfg.E, 128, scratch_bytes=4 * cfg.E * ctas)
    for a, b in zip(full, part):
        assert np.array_equal(np.asarray(a), np.asarray(b))


def test_dispatch_skewed_all_one_expert(M):
    T, K, E = 5000, 1, 3
    idx = np.full((T, K), 2, dtype=np.int32)
    cnt, blk, slot, src, st = _dispatch(M, idx, E, 128)
    ref = O.route(idx, E, 128)
    assert np.array_equal(slot, ref["slot"]) and list(cnt) == [0, 0, T]


@pytest.mark.parametrize("T", [512, 513])
def test_dispatch_single_cta_boundary(M, T):
    """4096 and 4104 pairs: the last full CTA chunk and one more CTA with a
    ragged 8-pair chunk; both give the oracle's routing."""
    rng = np.random.default_rng(7 + T)
    E, K = 96, 8
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[rng.random(idx.shape) < 0.03] = -1
    cnt, blk, slot, src, st = _dispatch(M, idx, E, 128)
    ref = O.route(idx, E, 128)
    assert st == 0
    assert np.array_equal(cnt, ref["cnt"]) and np.array_equal(blk, ref["blk_off"])
    assert np.array_equal(slot, ref["slot"])
    assert np.array_equal(src[:len(ref["src"])], ref["src"])


def test_dispatch_flags_out_of_range_experts_many_ctas(M):
    """An out-of-range index in the middle CTA of a 12-CTA dispatch is flagged."""
    rng = np.random.default_rng(11)
    T, K, E = 3000, 2, 50
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    idx[1234, 1] = E + 3
    cnt, blk, slot, src, st = _dispatch(M, idx, E, 64)
    ref = O.route(idx, E, 64)
    assert st == M.MM_MOE_ERR_BAD_ROUTING
    assert np.array_equal(slot, ref["slot"]) and np.array_equal(cnt, ref["cnt"])
