"""Shared helpers of the GPU parity tests: run the library through its C ABI on
seeded workload inputs, run the oracle on the same bytes, apply the criteria."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import workload as W


def calc_diff(x, y) -> float:
    """1 - 2<x,y> / (|x|^2 + |y|^2) in fp64 (DeepGEMM's calc_diff)."""
    x = np.asarray(x, dtype=np.float64).ravel()
    y = np.asarray(y, dtype=np.float64).ravel()
    den = float(np.dot(x, x) + np.dot(y, y))
    return 0.0 if den == 0 else 1.0 - 2.0 * float(np.dot(x, y)) / den


def check_output(got: np.ndarray, ref: np.ndarray, label: str = "") -> dict:
    """Criteria: calc_diff <= 1e-4 and every |got - ref| <= 2e-2 x that row's RMS
    (rows whose reference is all zero must be exactly zero)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    cd = calc_diff(got, ref)
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    err = np.abs(got - ref)
    ratio = np.where(rms > 0, err / np.where(rms > 0, rms, 1), np.where(err > 0, np.inf, 0))
    worst = float(ratio.max()) if ratio.size else 0.0
    assert cd <= 1e-4, f"{label}: calc_diff {cd:.3e} > 1e-4"
    assert worst <= 2e-2, f"{label}: max |err|/row_rms {worst:.3e} > 2e-2"
    return {"calc_diff": cd, "max_err_over_rms": worst}


def to_dev(inp: dict, device="cuda") -> dict:
    return {k: v.to(device) for k, v in inp.items()}


def run_forward(M, cfg, dev_inp: dict, opt=None, ws=None, out=None, prepared=None):
    """One forward through the C ABI (with cfg.S shared experts).  Returns (out, ws, prepared, status)."""
    opt = opt or M.options(M.MM_MOE_VARIANT_MX if cfg.variant == "mx" else M.MM_MOE_VARIANT_F8)
    opt.shared_experts = cfg.S
    if prepared is None:
        prepared = M.prepare_weights(dev_inp["w1_sf"], dev_inp["w2_sf"], cfg.H, cfg.I, cfg.E + cfg.S, opt)
    if ws is None:
        ws = M.alloc_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, opt)
    if out is None:
        out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    M.forward(dev_inp["x"], dev_inp["x_sf"], dev_inp["topk_idx"], dev_inp["topk_w"], dev_inp["w1"], prepared[0],
              dev_inp["w2"], prepared[1], out, cfg.H, cfg.I, cfg.E, ws, opt)
    status = M.sync_status(ws)
    return out, ws, prepared, status


def host_experts(dev_inp: dict):
    """Per-expert host copies of the (device) weights, fetched lazily for the oracle."""
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = tuple(dev_inp[k][e].cpu().numpy() for k in ("w1", "w1_sf", "w2", "w2_sf"))
        return cache[e]
    return get


def f8_gran(cfg, opt=None) -> int:
    """The FP8 intermediate's scale width a call uses: 128 by default, the oracle's
    shape rule for -1, else the pinned width."""
    g = int(opt.f8_act_gran) if opt is not None else 0
    return O.f8_act_gran(cfg.H, cfg.I) if g == -1 else (g or 128)


def oracle_rows(cfg, dev_inp: dict, rows, keep_intermediate=True, partials_bf16=False, clamp=None, f8_gran=128):
    x = dev_inp["x"].cpu().numpy()
    x_sf = dev_inp["x_sf"].cpu().numpy()
    idx = dev_inp["topk_idx"].cpu().numpy()
    w = dev_inp["topk_w"].cpu().numpy()
    return O.forward(rows, x, x_sf, idx, w, host_experts(dev_inp), cfg.H, cfg.I, cfg.E, cfg.variant,
                     keep_intermediate=keep_intermediate, partials_bf16=partials_bf16, clamp=clamp,
                     f8_gran=f8_gran, shared=cfg.S)


# Lines printed in pytest's terminal summary (tests/conftest.py): what the
# intermediate comparisons measured, so that a passing run still reports them.
REPORT = []

# FP8 scale agreement: s = fp32(amax / 448) moves with amax, and the GPU's amax
# comes from fp32 tensor-core partials promoted in fp32 over H/128 k-blocks,
# the oracle's from fp64 sums rounded once to fp32.  Measured on GB300 over the
# full-size FP8 rows: median 1, 99.9th percentile 8, max 12 fp32 ulps apart.
# Two scales count as the same scale when they are at most 16 ulps apart;
# every code of a block beyond that counts as a mismatch.
F8_SCALE_ULPS = 16


def intermediate_match(M, cfg, ws, opt, slot: np.ndarray, inter: dict, label: str = "") -> float:
    """Fraction of intermediate e4m3 codes equal (by value) to the oracle's, with
    every code of a block whose scale differs counted as a mismatch.  MX scales
    are UE8M0 bytes and must be equal; FP8 scales are raw fp32 amax/448 and must
    be within F8_SCALE_ULPS (the fp32 accumulation's spread, above).  The match
    fraction and, for FP8, the scale deviations in fp32 ulps are recorded in
    REPORT."""
    rows = int(M.mm_moe_workspace_region(ws.data_ptr(), opt, cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, 4)[1] // 4)
    codes = torch.empty(rows, cfg.I, dtype=torch.uint8, device="cuda")
    bs = 32 if cfg.variant == "mx" else f8_gran(cfg, opt)
    sf = torch.empty(rows, cfg.I // bs, dtype=torch.uint8 if cfg.variant == "mx" else torch.float32, device="cuda")
    r = M.mm_moe_read_intermediate(ws.data_ptr(), opt, cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, rows, codes.data_ptr(),
                                   sf.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert r == 0
    torch.cuda.synchronize()
    codes = codes.cpu().numpy()
    sf = sf.cpu().numpy()
    total = match = 0
    ulps = []
    for (t, k), (oc, osf) in inter.items():
        row = int(slot[t, k])
        assert row >= 0
        if cfg.variant == "mx":
            same_sf = np.repeat(sf[row] == osf, bs)
        else:
            g = sf[row].astype(np.float32)
            r = np.asarray(osf, dtype=np.float32)
            # distance in fp32 ulps of the oracle's scale (positive normal floats: integer bit distance)
            d = np.abs(g.view(np.int32).astype(np.int64) - r.view(np.int32).astype(np.int64))
            ulps.append(d)
            same_sf = np.repeat(d <= F8_SCALE_ULPS, bs)
        same = same_sf & (O.e4m3_decode(codes[row]) == O.e4m3_decode(oc))
        total += same.size
        match += int(same.sum())
    frac = match / max(total, 1)
    line = f"{label or cfg.name}: intermediate codes {match}/{total} equal ({100 * frac:.4f} %)"
    if ulps:
        u = np.concatenate(ulps)
        line += (f"; fp32 scale distance in ulps: median {np.median(u):.0f}, 99.9 % {np.percentile(u, 99.9):.0f}, "
                 f"max {u.max()}, blocks within {F8_SCALE_ULPS} ulps {100 * np.mean(u <= F8_SCALE_ULPS):.3f} %")
    REPORT.append(line)
    return frac


def read_routing(M, cfg, ws, opt):
    cnt = torch.empty(cfg.E + cfg.S, dtype=torch.int32, device="cuda")      # shared experts included
    blk = torch.empty(cfg.E + cfg.S + 1, dtype=torch.int32, device="cuda")
    slot = torch.empty(cfg.T, cfg.K + cfg.S, dtype=torch.int32, device="cuda")
    nsrc = M.mm_moe_workspace_region(ws.data_ptr(), opt, cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, 4)[1] // 4
    src = torch.empty(nsrc, dtype=torch.int32, device="cuda")
    r, bm = M.mm_moe_read_routing(ws.data_ptr(), opt, cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cnt.data_ptr(),
                                  blk.data_ptr(), slot.data_ptr(), src.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert r == 0
    torch.cuda.synchronize()
    return cnt.cpu().numpy(), blk.cpu().numpy(), slot.cpu().numpy(), src.cpu().numpy(), bm
