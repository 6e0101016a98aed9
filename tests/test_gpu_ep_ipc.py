"""Expert parallelism across processes: one process per rank, each holding only
its own tokens and buffers, the peers' buffers mapped by CUDA IPC
(`ep.share_peers`), the counts all-gathered and the steps separated by a device
synchronisation plus a gloo barrier (`ep.forward_distributed`).  The ranks share
one GPU here; no kernel waits for another process.  Each rank's output must equal,
bit for bit, its rows of the single-process forward with bf16 partials over all
tokens (the EP combine receives every pair's output as bf16), with the push and
the pull combine and with receive buffers sized by a token bound."""
import os
import socket
import traceback

import pytest
import torch

import workload as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_expert_forward_gb300 import build
    build.build()       # in-tree, before the rank processes load it


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, N, port, cfg_kw, combine, bound, result_dir, splits):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    path = os.path.join(result_dir, f"rank{rank}.txt")
    try:
        from datetime import timedelta

        import torch.distributed as dist
        torch.cuda.set_device(0)
        dist.init_process_group("gloo", rank=rank, world_size=N, init_method=f"tcp://127.0.0.1:{port}",
                                timeout=timedelta(seconds=120))
        import moe_expert_forward_gb300 as M
        from moe_expert_forward_gb300 import ep
        from gpu_util import run_forward, to_dev
        cfg = W.Config(**cfg_kw)
        dev = to_dev(W.make_inputs(cfg, "cpu"))         # every rank generates the same seeded workload
        lo = sum(splits[:rank])                          # this rank's tokens, rank-major
        sl = slice(lo, lo + splits[rank])
        variant = M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8
        st = ep.RankState(rank, dev["x"][sl].contiguous(), dev["x_sf"][sl].contiguous(),
                          dev["topk_idx"][sl].contiguous(), dev["topk_w"][sl].contiguous(), cfg.E, N, variant)
        out, (send_row, rows, rex) = ep.forward_distributed(st, dev["w1"], dev["w1_sf"], dev["w2"], dev["w2_sf"],
                                                             cfg.I, combine=combine, num_tokens_bound=bound)
        single, _, _, (code, _) = run_forward(M, cfg, dev, M.options(variant, partials_bf16=1))
        same = code == 0 and torch.equal(out, single[sl])
        diff = float((out.float() - single[sl].float()).abs().max()) if out.numel() else 0.0
        dist.barrier()
        dist.destroy_process_group()
        with open(path, "w") as f:
            f.write(f"ok {int(same)} rows {rows} diff {diff}\n")
    except Exception:
        with open(path, "w") as f:
            f.write("error\n" + traceback.format_exc())


def _run(cfg, N, combine="push", bound=None, tmp_path=None, splits=None):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = _free_port()
    cfg_kw = dict(name=cfg.name, T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, variant=cfg.variant, seed=cfg.seed)
    splits = splits or [cfg.T // N] * N
    procs = [ctx.Process(target=_rank_main, args=(r, N, port, cfg_kw, combine, bound, str(tmp_path), splits))
             for r in range(N)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():          # only this test's own children, by handle
            p.kill()
            p.join()
    res = []
    for r in range(N):
        f = tmp_path / f"rank{r}.txt"
        assert f.exists(), f"rank {r} wrote no result (exit code {procs[r].exitcode})"
        text = f.read_text()
        assert text.startswith("ok "), text
        res.append(text.split())
    return res


CFGS = [W.Config("ipc_mx", T=256, H=512, I=256, E=8, K=3, seed=91),
        W.Config("ipc_f8", T=256, H=512, I=256, E=8, K=2, variant="f8", seed=92)]


@pytest.mark.parametrize("cfg", CFGS, ids=[c.name for c in CFGS])
def test_ep_two_processes_equal_single_gpu(cfg, tmp_path):
    res = _run(cfg, 2, tmp_path=tmp_path)
    for r, parts in enumerate(res):
        assert parts[1] == "1", f"rank {r}: {' '.join(parts)}"
        assert int(parts[3]) > 0


def test_ep_two_processes_pull_combine_with_bound(tmp_path):
    cfg = CFGS[0].with_(seed=93)
    res = _run(cfg, 2, combine="pull", bound=cfg.T // 2, tmp_path=tmp_path)
    for r, parts in enumerate(res):
        assert parts[1] == "1", f"rank {r}: {' '.join(parts)}"


def test_ep_two_processes_rank_without_tokens(tmp_path):
    """Rank 1 holds no tokens: it still owns half of the experts, receives rank
    0's pairs for them, and shares empty token buffers."""
    cfg = CFGS[0].with_(seed=94)
    res = _run(cfg, 2, tmp_path=tmp_path, splits=[cfg.T, 0])
    for r, parts in enumerate(res):
        assert parts[1] == "1", f"rank {r}: {' '.join(parts)}"
    assert int(res[1][3]) > 0


def _context_main(rank, N, port, cfg_kw, result_dir):
    """Two forwards through one ep.EPRank per process: the buffers and the peers'
    addresses are set up once; the second batch moves the tokens (rolled by 37,
    a fifth of the slots masked) and splits them unevenly."""
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    path = os.path.join(result_dir, f"rank{rank}.txt")
    try:
        from datetime import timedelta

        import torch.distributed as dist
        torch.cuda.set_device(0)
        dist.init_process_group("gloo", rank=rank, world_size=N, init_method=f"tcp://127.0.0.1:{port}",
                                timeout=timedelta(seconds=120))
        import moe_expert_forward_gb300 as M
        from moe_expert_forward_gb300 import ep
        from gpu_util import run_forward, to_dev
        cfg = W.Config(**cfg_kw)
        a = to_dev(W.make_inputs(cfg, "cpu"))
        b = {k: (torch.roll(v, 37, 0) if k in ("x", "x_sf", "topk_idx", "topk_w") else v) for k, v in a.items()}
        g = torch.Generator().manual_seed(cfg.seed + 1)
        b["topk_idx"] = torch.where(torch.rand(b["topk_idx"].shape, generator=g).cuda() < 0.2, -1, b["topk_idx"])
        variant = M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8
        bound = cfg.T // N + 24
        ctx = ep.EPRank(rank, N, cfg.E, cfg.K, cfg.H, cfg.I, variant, bound, a["w1"], a["w1_sf"], a["w2"],
                        a["w2_sf"], "cuda")
        ok = []
        for inp, splits, combine in ((a, [cfg.T // N] * N, "push"), (b, [cfg.T // N + 24, cfg.T // N - 24], "pull")):
            lo = sum(splits[:rank])
            sl = slice(lo, lo + splits[rank])
            out, _ = ctx.forward(inp["x"][sl].contiguous(), inp["x_sf"][sl].contiguous(),
                                 inp["topk_idx"][sl].contiguous(), inp["topk_w"][sl].contiguous(), combine=combine)
            single, _, _, (code, _) = run_forward(M, cfg, inp, M.options(variant, partials_bf16=1))
            ok.append(int(code == 0 and torch.equal(out, single[sl])))
        ctx.close()
        dist.barrier()
        dist.destroy_process_group()
        with open(path, "w") as f:
            f.write(f"ok {min(ok)} calls {len(ok)}\n")
    except Exception:
        with open(path, "w") as f:
            f.write("error\n" + traceback.format_exc())


@pytest.mark.parametrize("cfg", CFGS, ids=[c.name for c in CFGS])
def test_ep_rank_context_runs_two_batches(cfg, tmp_path):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = _free_port()
    cfg_kw = dict(name=cfg.name, T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, variant=cfg.variant, seed=cfg.seed)
    procs = [ctx.Process(target=_context_main, args=(r, 2, port, cfg_kw, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
    for r in range(2):
        f = tmp_path / f"rank{r}.txt"
        assert f.exists(), f"rank {r} wrote no result (exit code {procs[r].exitcode})"
        text = f.read_text()
        assert text.startswith("ok 1 "), text
