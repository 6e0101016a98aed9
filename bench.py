"""Benchmark of the MoE-layer forward on GB300 (one JSON line on rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config pro] [--impl ours|reference]

A step is one forward of one MoE layer (dispatch, gather, L1 GEMM + SwiGLU +
requant, L2 GEMM, combine) over one batch of T tokens of the named workload,
inputs resident in HBM.  The L2 cache is flushed (a 512 MiB write) between
timed steps, outside the timed events.  Per-kernel times come from CUDA events
the library records between its kernels on the launching stream.

--impl reference times the CPU oracle (fp64 numpy) on the host cores on a
bounded token sample of the same workload; it is the slow reference arm.

Under torchrun with N > 1 every rank runs an independent replica of the
workload (weak scaling; tokens are independent, so there is no collective on
the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workload as W  # noqa: E402

FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0          # nominal dense ratio (4.5 / 2.25 PFLOP/s)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


# ------------------------------------------------------------------ distributed (replicas only)
def dist_setup(n):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.start_wall = time.time()

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for ln in out.strip().splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append({"sm": float(f[1]), "max": float(f[2]), "power": float(f[3]),
                             "hw": f[5], "hwt": f[6], "swt": f[7], "pcap": f[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        # samples are ~100 ms apart; keep those taken while the GPU was busy (highest power third)
        pw = np.array([r["power"] for r in rows])
        busy = [r for r in rows if r["power"] >= np.percentile(pw, 66)] or rows
        reasons = set()
        for r in busy:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": float(np.median([r["sm"] for r in busy])), "sm_max_mhz": busy[0]["max"],
                "reasons": sorted(reasons), "samples": len(busy), "power_w_max": float(pw.max())}


# ------------------------------------------------------------------ accounting
def workload_accounting(cfg, idx: np.ndarray, part_elem: int = 4, x_bf16: bool = False):
    """Bytes / FLOPs of one step.  step_bytes is the method's algorithmic traffic:
    the weights + scales of every expert that receives a token, x + its scales,
    topk_idx + topk_w and the bf16 output.  The *_impl_bytes figures add this
    implementation's own traffic (pool rows, intermediate, partials) and are
    reported beside it, never in place of it (part_elem: bytes of one L2
    partial, 4 for fp32, 2 for bf16; x_bf16: the caller's x is bf16 and the
    gather quantises it)."""
    T, H, I, E, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K
    valid = (idx >= 0) & (idx < E)
    touched = int(np.unique(idx[valid]).size) + cfg.S      # shared experts: touched by every token
    pairs = int(valid.sum()) + T * cfg.S
    if cfg.variant == "mx":
        w1_b = 2 * I * H * (0.5 + 1 / 32)
        w2_b = H * I * (0.5 + 1 / 32)
        x_b = H * (1 + 1 / 32)
        a_b = I * (1 + 1 / 32)
    else:
        w1_b = 2 * I * H + (2 * I // 128) * (H // 128) * 4
        w2_b = H * I + (H // 128) * (I // 128) * 4
        x_b = H + (H // 128) * 4
        a_b = I + (I // 128) * 4
    x_in = 2 * H if x_bf16 else x_b          # the caller's row of x
    step_bytes = touched * (w1_b + w2_b) + T * x_in + T * K * 8 + T * H * 2
    flops = 6.0 * pairs * H * I
    # algorithmic bytes of the separate GEMM launches: their weight streams (+ x for L1)
    l1_bytes = touched * w1_b + T * x_in + T * K * 8
    l2_bytes = touched * w2_b
    # this implementation's own traffic on top of the algorithmic bytes
    impl = {"pool_rows_write_read": 2 * pairs * x_b, "intermediate_write_read": 2 * pairs * a_b,
            "partials_write_read": 2 * pairs * H * part_elem}
    return {"touched_experts": touched, "pairs": pairs, "step_bytes": step_bytes, "flops": flops,
            "l1_bytes": l1_bytes, "l2_bytes": l2_bytes, "impl_bytes": impl,
            "l1_flops": 4.0 * pairs * H * I, "l2_flops": 2.0 * pairs * H * I}


def kernel_traffic(kernel: str, cfg_name: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source (hash match); else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(f"{kernel}:{cfg_name}")
    if not ent:
        return None
    src = os.path.join(ROOT, "moe_expert_forward_gb300", "csrc", ent.get("source", "gemm_mx.cu"))
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return ent["dram_bytes_per_launch"] if h == ent.get("source_sha") else None


# ------------------------------------------------------------------ our arm
def run_ours(args, ws_n, rank, local):
    from moe_expert_forward_gb300 import build as B
    B.build()
    import moe_expert_forward_gb300 as M

    cfg = W.CONFIGS[args.config].with_(S=args.shared)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = W.make_inputs(cfg, dev)
    opt = M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8)
    opt.shared_experts = cfg.S
    opt.f8_act_gran = args.f8_gran
    if args.fused is not None:
        opt.fused = args.fused
    opt.partials_bf16 = 1 if args.partials == "bf16" else 0
    if args.early_combine is not None:
        opt.early_combine = args.early_combine
    if args.swap_ab is not None:
        opt.swap_ab = args.swap_ab
    if args.block_m:
        opt.block_m = args.block_m
    opt.ring_blocks = args.ring_blocks
    opt.lag_units = args.lag
    if args.x == "bf16":
        # bf16 activations: the gather quantises each row (x_sf is not read)
        inp["x"], inp["x_sf"] = W.make_x_bf16(cfg, dev), None
        opt.x_bf16 = 1
    fused = bool(opt.fused) and cfg.variant == "mx"
    w1p, w2p = M.prepare_weights(inp["w1_sf"], inp["w2_sf"], cfg.H, cfg.I, cfg.E + cfg.S, opt)
    ws = M.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, opt, dev)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def fwd(o, x=None, x_sf=None, idx=None, w=None, dst=None):
        M.forward(inp["x"] if x is None else x, inp["x_sf"] if x_sf is None else x_sf,
                  inp["topk_idx"] if idx is None else idx, inp["topk_w"] if w is None else w,
                  inp["w1"], w1p, inp["w2"], w2p, out if dst is None else dst, cfg.H, cfg.I, cfg.E, ws, o)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        fwd(opt)
    code, where = M.sync_status(ws)
    if code != 0:
        raise RuntimeError(f"device status {code} at site {where}")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(M.MM_MOE_NUM_TIMING_EVENTS)] for _ in range(K)]
    for row in evs:                  # torch creates the CUDA event on first record
        for e in row:
            e.record()
    torch.cuda.synchronize()
    import ctypes
    # the timed steps record only their first and last event: an event between two
    # kernels would keep the library from launching the second one programmatically
    edge = lambda row: [row[0].cuda_event] + [None] * (M.MM_MOE_NUM_TIMING_EVENTS - 2) + [row[-1].cuda_event]
    arrays = [(ctypes.c_void_p * M.MM_MOE_NUM_TIMING_EVENTS)(*edge(row)) for row in evs]
    assert all(arr[0] and arr[-1] for arr in arrays)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier(ws_n)
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        o = M.mm_moe_options.from_buffer_copy(opt)
        o.timing_events = ctypes.cast(arrays[i], ctypes.c_void_p)
        fwd(o)
    torch.cuda.synchronize()
    barrier(ws_n)
    code, where = M.sync_status(ws)
    if code != 0:
        raise RuntimeError(f"device status {code} at site {where}")
    step_ms_local = float(np.mean([evs[i][0].elapsed_time(evs[i][-1]) for i in range(K)]))
    step_ms = max_over_ranks(step_ms_local, ws_n)
    # the stage breakdown: a few more steps with every event recorded (no programmatic launches)
    n_st = 3
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(M.MM_MOE_NUM_TIMING_EVENTS)] for _ in range(n_st)]
    for row in sev:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    sarr = [(ctypes.c_void_p * M.MM_MOE_NUM_TIMING_EVENTS)(*[e.cuda_event for e in row]) for row in sev]
    for i in range(n_st):
        flush.zero_()
        o = M.mm_moe_options.from_buffer_copy(opt)
        o.timing_events = ctypes.cast(sarr[i], ctypes.c_void_p)
        fwd(o)
    torch.cuda.synchronize()
    stage_ms = np.array([[sev[i][j].elapsed_time(sev[i][j + 1]) for j in range(5)] for i in range(n_st)])

    # optional per-task trace of one more step (the kernel's timing instantiation, after the timed steps)
    trace_summary = None
    if args.trace and cfg.variant == "mx" and not opt.swap_ab:
        from moe_expert_forward_gb300 import trace as TR
        launches = 1 if fused else 2
        tbuf = torch.zeros(TR.buffer_bytes(torch.cuda.get_device_properties(dev).multi_processor_count, 4096,
                                           launches), dtype=torch.uint8, device=dev)
        o = M.mm_moe_options.from_buffer_copy(opt)
        o.trace_buf, o.trace_bytes = tbuf.data_ptr(), tbuf.numel()
        flush.zero_()
        fwd(o)
        torch.cuda.synchronize()
        trace_summary = TR.summary(TR.records(tbuf))
        del tbuf

    # end to end, as a serving loop runs it: every step copies its inputs from pinned host
    # memory and reads its output back to pinned host memory.  The copies run on streams of
    # their own with two buffer sets, so step i+1's inputs and step i-1's output move while
    # step i computes; the value is the steps over the wall time from the first timed copy
    # to the last.  No L2 flush here: each step reads >= 2.5 GB of weights, far more than
    # L2, and its inputs arrive fresh by copy.
    host = {k: inp[k].cpu().pin_memory() for k in ("x", "x_sf", "topk_idx", "topk_w") if inp[k] is not None}
    nbuf = 2
    dbuf = [{k: torch.empty_like(inp[k]) for k in host} for _ in range(nbuf)]
    douts = [torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    houts = [torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = houts[0].numel() * houts[0].element_size()
    # three streams of their own (the default, legacy stream would serialise against the
    # copies): inputs in, compute, output out.  One copy stream would queue step i+1's
    # inputs behind step i's read-back, which waits for step i's forward.
    cs, hs, ds = (torch.cuda.Stream(device=dev) for _ in range(3))
    e2e_warm, e2e_n = 3, max(3, min(K, 50))
    total = e2e_warm + e2e_n
    ev_in = [torch.cuda.Event() for _ in range(total)]
    ev_fw = [torch.cuda.Event() for _ in range(total)]
    ev_out = [torch.cuda.Event() for _ in range(total)]
    t_first, t_last = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for i in range(total):
        j = i % nbuf
        if i == e2e_warm:
            torch.cuda.synchronize()                 # the timed steps start from an idle GPU: fill and drain count
        with torch.cuda.stream(hs):
            if i >= nbuf:
                hs.wait_event(ev_fw[i - nbuf])       # input set j: its last forward has read it
            if i == e2e_warm:
                t_first.record(hs)
            for k in host:
                dbuf[j][k].copy_(host[k], non_blocking=True)
            ev_in[i].record(hs)
        with torch.cuda.stream(cs):
            cs.wait_event(ev_in[i])
            if i >= nbuf:
                cs.wait_event(ev_out[i - nbuf])        # output buffer j: its last read-back is done
            fwd(opt, dbuf[j]["x"], dbuf[j].get("x_sf"), dbuf[j]["topk_idx"], dbuf[j]["topk_w"], douts[j])
            ev_fw[i].record(cs)
        with torch.cuda.stream(ds):
            ds.wait_event(ev_fw[i])
            houts[j].copy_(douts[j], non_blocking=True)
            ev_out[i].record(ds)
    with torch.cuda.stream(ds):
        t_last.record(ds)
    torch.cuda.synchronize()
    code, _ = M.sync_status(ws)
    assert code == 0
    assert torch.equal(houts[(total - 1) % nbuf], douts[(total - 1) % nbuf].cpu())
    assert torch.equal(douts[(total - 1) % nbuf], out)   # the same inputs give the device-timed output
    e2e_ms = [t_first.elapsed_time(t_last) / e2e_n]
    e2e_step_ms = max_over_ranks(float(np.mean(e2e_ms)), ws_n)
    clk = clocks.stop()

    idx_np = inp["topk_idx"].cpu().numpy()
    acc = workload_accounting(cfg, idx_np, 2 if opt.partials_bf16 else 4, bool(opt.x_bf16))
    pk, pk_src = peaks()
    hbm = float(pk["hbm_gbs"])
    fp8 = float(pk["bf16_tflops"]) * FP8_OVER_BF16
    stage_mean = stage_ms.mean(0)
    l1_ms, l2_ms = float(stage_mean[2]), float(stage_mean[3])
    early = fused and bool(opt.early_combine)
    if fused:
        # one launch runs gather, L1 and L2: the layer's algorithmic bytes all pass through it
        # (the bf16 output is counted too, although the combine kernel after it writes that)
        dom, dom_ms = "fused", l1_ms + l2_ms
        dom_bytes = acc["step_bytes"]
        dom_flops = acc["flops"]
    else:
        # dominant kernel: the one with the largest share of the step
        dom = "l1" if l1_ms >= l2_ms else "l2"
        dom_ms = l1_ms if dom == "l1" else l2_ms
        dom_bytes = acc["l1_bytes"] if dom == "l1" else acc["l2_bytes"]
        dom_flops = acc["l1_flops"] if dom == "l1" else acc["l2_flops"]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    t_roof = max(acc["flops"] / (fp8 * 1e12), acc["step_bytes"] / (hbm * 1e9))
    tokens_per_s = ws_n * cfg.T / (step_ms * 1e-3)

    result = {
        "metric": "MoE-layer tokens/s (one MoE layer forward, 1 GPU per replica)",
        "value": tokens_per_s,
        "unit": "tokens/s",
        "n_gpus": ws_n,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3xe2m1->fp32acc" if cfg.variant == "mx" else "e4m3xe4m3->fp32acc",
        "data": "synthetic (seeded workload generator; random weights, no checkpoint)",
        "config": {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} top-{cfg.K} "
                               f"{'uniform' if cfg.routing == 'uniform' else 'Zipf(1.1)'} routing, "
                               f"{'MX e4m3 x e2m1 UE8M0/32' if cfg.variant == 'mx' else 'FP8 e4m3 per-128'}",
                   "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "K": cfg.K, "seed": cfg.seed,
                   "l2_policy": "L2 flushed (512 MiB write) before every timed step; weights 3+ GB >> L2",
                   "parallelism": f"replicas x{ws_n} (no data-path collective)",
                   "fused_stream": fused, "early_combine": early, "partials": args.partials, "x": args.x,
                   "swap_ab": int(opt.swap_ab), "block_m": int(opt.block_m),
                   "shared_experts": cfg.S, "f8_act_gran": int(opt.f8_act_gran),
                   "ring_blocks": int(opt.ring_blocks), "lag_units": int(opt.lag_units),
                   "e2e_policy": "copies on streams of their own, two buffer sets (step i+1 in and step i-1 out "
                                 "overlap step i); no L2 flush: every step reads >= 2.5 GB of weights"},
        "tflops": acc["flops"] / (step_ms * 1e-3) / 1e12,
        "path_roofline": {"t_roofline_us": t_roof * 1e6, "frac": t_roof / (step_ms * 1e-3),
                          "bytes": acc["step_bytes"], "flops": acc["flops"],
                          "touched_experts": acc["touched_experts"],
                          "peaks": {"hbm_gbs": hbm, "fp8_tflops": fp8, "source": pk_src,
                                    "fp8_from": "bf16_tflops x 2 (nominal fp8/bf16 ratio)"}},
        "stages_ms": ({"dispatch": float(stage_mean[0]), "fused_gather_l1_l2": float(stage_mean[2] + stage_mean[3]),
                       "combine": float(stage_mean[4])} if fused else
                      {s: float(v) for s, v in zip(M.STAGES, stage_mean)}),
        "roofline": {"kernel": (f"gemm_mx_kernel (fused gather + L1 + L2{' + combine' if early else ''} stream)" if fused else
                                f"gemm_{'mx' if cfg.variant == 'mx' else 'f8'}_kernel ({dom.upper()} grouped GEMM)"),
                     "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": kernel_traffic(dom, cfg.name if args.partials == "fp32" else f"{cfg.name}:bf16-partials"),
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "algorithmic_bytes_def": ("weights + scales of the touched experts, x + x_sf, topk_idx + topk_w, "
                                               "bf16 out" if fused else
                                               ("W1 + scales of the touched experts, x + x_sf, topk" if dom == "l1"
                                                else "W2 + scales of the touched experts")),
                     "launch_ms": dom_ms,
                     "implementation_bytes_per_launch": (
                         {k: v for k, v in acc["impl_bytes"].items()} if fused else None),
                     "tensor_frac": dom_flops / (dom_ms * 1e-3) / (fp8 * 1e12),
                     "peak_source": f"{pk_src} hbm_gbs (STREAM-style copy); tensor_frac against "
                                    f"2 x {pk_src} bf16_tflops (nominal fp8/bf16 ratio)"},
        "e2e": {"value": ws_n * cfg.T / (e2e_step_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_step_ms},
        "gpu_launches": (3 if early else (4 if fused else 6)) * K,   # dispatch x2, [gather], GEMM(s), [combine]
        "clocks": clk,
    }
    if trace_summary is not None:
        result["trace"] = trace_summary
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, inp, args.cpu_tokens or CPU_TOKENS[cfg.name], args.f8_gran)
    return result


# ------------------------------------------------------------------ oracle (CPU) runs
# tokens the oracle baseline times once per workload: about 10-30 s of host work each
CPU_TOKENS = {"tiny": 64, "flash": 16, "pro": 4, "decode": 16, "f8": 8, "pro96": 4, "f8x": 8}


def oracle_tokens(cfg, inp, rows, f8_opt=0):
    """Times the oracle on `rows`; f8_opt is the f8_act_gran option (0: per 128,
    -1: the pages' shape rule, else the width)."""
    import oracle as O
    f8_gran = O.f8_act_gran(cfg.H, cfg.I) if f8_opt == -1 else (f8_opt or 128)
    bf16_x = inp["x_sf"] is None             # the layer quantises bf16 rows first: the oracle does too
    x = inp["x"][rows].float().cpu().numpy() if bf16_x else inp["x"][rows].cpu().numpy()
    x_sf = None if bf16_x else inp["x_sf"][rows].cpu().numpy()
    idx = inp["topk_idx"][rows].cpu().numpy()
    w = inp["topk_w"][rows].cpu().numpy()
    cache = {}

    def experts(e):
        if e not in cache:
            cache[e] = tuple(inp[k][e].cpu().numpy() for k in ("w1", "w1_sf", "w2", "w2_sf"))
        return cache[e]
    # fetch the weights first so that only the oracle's arithmetic is timed
    for e in list(np.unique(idx[(idx >= 0) & (idx < cfg.E)])) + list(range(cfg.E, cfg.E + cfg.S)):
        experts(int(e))
    t0 = time.perf_counter()
    c0 = time.process_time()
    if bf16_x:
        x, x_sf = O.quantise_x(x, cfg.variant)
    O.forward(range(len(rows)), x, x_sf, idx, w, experts, cfg.H, cfg.I, cfg.E, cfg.variant,
              f8_gran=f8_gran, shared=cfg.S)
    dt = time.perf_counter() - t0
    return dt, (time.process_time() - c0) / dt


def blas_threads() -> str:
    """numpy's BLAS thread setting as the environment fixes it (unset: the library's default)."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return f"{var}={os.environ[var]}"
    return "unset (numpy's BLAS default)"


def cpu_baseline(cfg, inp, n_tokens, f8_opt=0):
    rows = list(range(min(n_tokens, cfg.T)))
    dt, busy = oracle_tokens(cfg, inp, rows, f8_opt)
    return {"value": len(rows) / dt, "unit": "tokens/s", "cores": round(busy, 2),
            "cores_available": len(os.sched_getaffinity(0)), "blas_threads": blas_threads(),
            "cores_def": "CPU seconds / wall seconds of the timed oracle call (the average number of "
                         "busy host threads)",
            "kind": "oracle", "sample": f"first {len(rows)} tokens of the {cfg.name} workload "
                                        f"({len(rows) * cfg.K} routed pairs), fp64 numpy, {dt:.1f} s",
            "full_T_extrapolated": {"seconds": dt * cfg.T / len(rows), "tokens_per_s": len(rows) / dt,
                                    "how": f"linear in tokens: {dt:.2f} s x {cfg.T} / {len(rows)} "
                                           f"(an extrapolation, not a measurement)"}}


def run_reference(args, ws_n, rank):
    cfg = W.CONFIGS[args.config].with_(S=args.shared)
    if rank != 0:
        return None
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = W.make_inputs(cfg, dev, with_weights=False)
    if args.x == "bf16":
        inp["x"], inp["x_sf"] = W.make_x_bf16(cfg, dev), None
    # only the experts the sampled tokens use are materialised
    n = args.ref_tokens
    rows = list(range(min(n, cfg.T)))
    used = sorted(set(int(e) for e in inp["topk_idx"][rows].cpu().numpy().ravel() if e >= 0))
    used += list(range(cfg.E, cfg.E + cfg.S))          # shared experts
    inp.update(W.make_weights(cfg, dev, experts=used))
    times, busy = [], []
    for i in range(max(args.warmup, 0) + args.steps):
        dt, b = oracle_tokens(cfg, inp, rows, args.f8_gran)
        if i >= args.warmup:
            times.append(dt)
            busy.append(b)
    step_s = float(np.mean(times))
    v = len(rows) / step_s
    cores = round(float(np.mean(busy)), 2)
    return {"impl": "reference", "metric": "MoE-layer tokens/s (one MoE layer forward, 1 GPU per replica)",
            "value": v, "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded workload generator)",
            "config": {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} top-{cfg.K}",
                       "sample_tokens": len(rows), "x": args.x},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores,
                             "cores_available": len(os.sched_getaffinity(0)), "blas_threads": blas_threads(),
                             "kind": "oracle",
                             "sample": f"first {len(rows)} tokens per step ({len(rows) * cfg.K} pairs)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="pro", choices=list(W.CONFIGS),
                    help="workload (default pro: the largest single-GPU configuration)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--partials", default="fp32", choices=["fp32", "bf16"],
                    help="L2 partials: fp32 (default) or cast to bf16 before the combine")
    ap.add_argument("--early-combine", type=int, choices=[0, 1], default=None,
                    help="fused stream: combine in the GEMM's epilogue warps (library default 1) or in a kernel after it")
    ap.add_argument("--x", default="fp8", choices=["fp8", "bf16"],
                    help="activations: fp8 codes + scales (default) or bf16, quantised inside the gather")
    ap.add_argument("--cpu-tokens", type=int, default=0,
                    help="tokens of the workload the oracle baseline times once (0: a per-workload count "
                         "sized for about 10-30 s of host work)")
    ap.add_argument("--ref-tokens", type=int, default=2,
                    help="--impl reference: tokens of the workload the oracle processes per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--swap-ab", type=int, choices=[0, 1, 2], default=None,
                    help="MX: 1 = weights as the MMA M side, each pool block tokens as N; 2 = the same on 2-CTA clusters; default: the library choice")
    ap.add_argument("--block-m", type=int, default=0, help="tokens per pool block (0: the library's choice)")
    ap.add_argument("--shared", type=int, default=0,
                    help="shared experts added to the workload (used by every token with weight 1)")
    ap.add_argument("--f8-gran", type=int, choices=[-1, 0, 64, 128], default=0,
                    help="FP8: intermediate scale width (0: per 128, the library default; -1: the pages' shape rule)")
    ap.add_argument("--ring-blocks", type=int, default=0,
                    help="MX fused stream: the intermediate as a ring of this many pool blocks (0: the whole pool)")
    ap.add_argument("--trace", action="store_true",
                    help="MX token-M kernel: trace one extra step per task and add its phase summary ('trace')")
    ap.add_argument("--lag", type=int, default=-1,
                    help="fused stream: experts by which L2 trails L1 (-1: the library's choice)")
    ap.add_argument("--fused", type=int, choices=[0, 1], default=None,
                    help="1: gather + L1 + L2 as one lag-ordered persistent launch; default: the library's")
    args = ap.parse_args()
    ws_n, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, ws_n, rank)
    else:
        res = run_ours(args, ws_n, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
