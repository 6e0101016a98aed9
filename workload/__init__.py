"""Seeded synthetic inputs for the MoE-layer forward (shared by tests, bench and smoke).

This module only *draws* inputs and puts them into the storage formats the
forward consumes (e4m3 / e2m1 codes with UE8M0 or fp32 block scales).  It holds
none of the forward's own arithmetic: no GEMM, no SwiGLU, no requantisation of
the intermediate activation, no combine.  Both the CUDA path and the CPU oracle
receive byte-identical copies of what it returns.

Workload recipe (shapes follow the DeepSeek-V4 Flash / Pro / MiMo-V2.5 MoE
shapes used by the MegaMoE pages' benchmarks; no dataset or trained weights):
  * routing: each token draws K distinct experts as the top-K of i.i.d. Gumbel
    keys (uniform), or of log p_r + Gumbel with p_r ~ r^-s over a seeded
    permutation of the experts (Zipf skew, decode shape);
  * topk_w = softmax of N(0,1) logits over the K chosen experts (fp32);
  * x ~ N(0,1) [T,H]; W1 ~ N(0,0.02) [E,2I,H] (rows [0,I) gate, [I,2I) up);
    W2 ~ N(0,0.02) [E,H,I];
  * MX format: x -> e4m3 with one UE8M0 scale per 1x32 along H; W -> e2m1
    (two per byte, low nibble = even index) with one UE8M0 scale per 1x32
    along the contraction dimension;
  * F8 format: x -> e4m3 with one fp32 scale per 1x128; W -> e4m3 with one
    fp32 scale per 128x128 block.
Each expert's weights come from their own sub-seed, so any expert can be
regenerated alone.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    variant: str = "mx"        # "mx": e4m3 x e2m1, UE8M0 per 32; "f8": e4m3 x e4m3, fp32 per 128
    routing: str = "uniform"   # "uniform" | "zipf"
    zipf_s: float = 1.1
    seed: int = 0
    S: int = 0                 # shared experts: experts E .. E+S-1, used by every token (not routed)

    @property
    def flops(self) -> float:
        """Routed-pair FLOPs of both grouped GEMMs: 2*T*K*H*(2I) + 2*T*K*I*H."""
        return 6.0 * self.T * self.K * self.H * self.I

    def with_(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS: Dict[str, Config] = {
    "tiny": Config("tiny", T=64, H=256, I=128, E=8, K=2, seed=0),
    "flash": Config("flash", T=2048, H=4096, I=2048, E=256, K=6, seed=1),
    "pro": Config("pro", T=8192, H=7168, I=3072, E=384, K=6, seed=2),
    "decode": Config("decode", T=128, H=4096, I=2048, E=256, K=8, routing="zipf", seed=3),
    "f8": Config("f8", T=8192, H=4096, I=2048, E=256, K=8, variant="f8", seed=4),
}
CONFIG_ORDER = ["tiny", "flash", "pro", "decode", "f8"]
# Reduced cases for hardware-counter captures: the pro-shaped and FP8-shaped
# workloads with fewer tokens and experts but the same tokens per expert (128
# and 256) and the same H, I and top-k, so that a multi-pass profile holds a few
# GB on the device.  They are not benchmark workloads.
CONFIGS["pro96"] = Config("pro96", T=2048, H=7168, I=3072, E=96, K=6, seed=2)
CONFIGS["f8x"] = Config("f8x", T=2048, H=4096, I=2048, E=64, K=8, variant="f8", seed=4)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


# ---------------------------------------------------------------- storage formats
def _ue8m0_exponent(amax: torch.Tensor, qmax_mant: float, qmax_exp: int) -> torch.Tensor:
    """Smallest integer e with qmax * 2^e >= amax, qmax = qmax_mant * 2^qmax_exp
    (qmax_mant in [0.5,1)), computed exactly from frexp; clamped to [-127,127]."""
    m, ex = torch.frexp(amax)
    e = torch.where(m <= qmax_mant, ex - qmax_exp, ex - qmax_exp + 1)
    return e.clamp(-127, 127).to(torch.int32)


def quant_e4m3_ue8m0(x: torch.Tensor, block: int = 32):
    """x [R,C] fp32 -> (codes u8 [R,C], sf u8 [R,C/block]), UE8M0 scale 2^e with
    e the smallest integer such that 448*2^e >= block amax."""
    R, C = x.shape
    xb = x.float().reshape(R, C // block, block)
    amax = xb.abs().amax(-1).clamp_min(1e-10)
    e = _ue8m0_exponent(amax, 0.875, 9)                  # 448 = 0.875 * 2^9
    scaled = xb * torch.exp2(-e.float()).unsqueeze(-1)   # exact (power of two)
    codes = scaled.to(torch.float8_e4m3fn).view(torch.uint8).reshape(R, C)
    return codes, (e + 127).to(torch.uint8)


def quant_e2m1_ue8m0(w: torch.Tensor, block: int = 32):
    """w [R,C] fp32 -> (packed u8 [R,C/2] low nibble = even column, sf u8 [R,C/block]).
    e2m1 magnitudes {0,.5,1,1.5,2,3,4,6}; round to nearest, ties to even code."""
    R, C = w.shape
    wb = w.float().reshape(R, C // block, block)
    amax = wb.abs().amax(-1).clamp_min(1e-10)
    e = _ue8m0_exponent(amax, 0.75, 3)                   # 6 = 0.75 * 2^3
    v = (wb * torch.exp2(-e.float()).unsqueeze(-1)).reshape(R, C)
    a = v.abs()
    mag = ((a > 0.25).int() + (a >= 0.75).int() + (a > 1.25).int() + (a >= 1.75).int()
           + (a > 2.5).int() + (a >= 3.5).int() + (a > 5.0).int())
    nib = torch.where((v < 0) & (mag > 0), mag + 8, mag).to(torch.uint8)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).contiguous()
    return packed, (e + 127).to(torch.uint8)


def quant_e4m3_f32_rows(x: torch.Tensor, block: int = 128):
    """x [R,C] -> (codes u8 [R,C], sf f32 [R,C/block]); sf = max(amax,1e-10)/448."""
    R, C = x.shape
    xb = x.float().reshape(R, C // block, block)
    sf = xb.abs().amax(-1).clamp_min(1e-10) / 448.0
    codes = (xb / sf.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8).reshape(R, C)
    return codes, sf.contiguous()


def quant_e4m3_f32_blocks(w: torch.Tensor, block: int = 128):
    """w [R,C] -> (codes u8 [R,C], sf f32 [R/block, C/block]) one scale per block x block."""
    R, C = w.shape
    wb = w.float().reshape(R // block, block, C // block, block)
    sf = wb.abs().amax(dim=(1, 3)).clamp_min(1e-10) / 448.0
    codes = (wb / sf[:, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(R, C)
    return codes, sf.contiguous()


# ---------------------------------------------------------------- routing
def make_routing(cfg: Config, device="cpu"):
    """topk_idx int32 [T,K] (K distinct experts per token), topk_w fp32 [T,K]."""
    g = _gen(cfg.seed, 0, device)
    u = torch.rand(cfg.T, cfg.E, generator=g, device=device, dtype=torch.float64)
    gumbel = -torch.log(-torch.log(u.clamp(1e-300, 1.0 - 1e-16)))
    if cfg.routing == "uniform":
        keys = gumbel
    elif cfg.routing == "zipf":
        gp = _gen(cfg.seed, 1, device)
        perm = torch.randperm(cfg.E, generator=gp, device=device)
        ranks = torch.empty(cfg.E, dtype=torch.float64, device=device)
        ranks[perm] = torch.arange(1, cfg.E + 1, dtype=torch.float64, device=device)
        keys = gumbel + (-cfg.zipf_s * torch.log(ranks))[None, :]
    else:
        raise ValueError(cfg.routing)
    idx = torch.topk(keys, cfg.K, dim=1).indices.to(torch.int32).contiguous()
    gl = _gen(cfg.seed, 2, device)
    logits = torch.randn(cfg.T, cfg.K, generator=gl, device=device, dtype=torch.float32)
    w = torch.softmax(logits, dim=1).contiguous()
    return idx, w


# ---------------------------------------------------------------- activations / weights
def make_x(cfg: Config, device="cpu"):
    g = _gen(cfg.seed, 3, device)
    x = torch.randn(cfg.T, cfg.H, generator=g, device=device, dtype=torch.float32)
    if cfg.variant == "mx":
        return quant_e4m3_ue8m0(x, 32)
    return quant_e4m3_f32_rows(x, 128)


def make_x_bf16(cfg: Config, device="cpu"):
    """bf16 activations [T, H] ~ N(0, 1) for the bf16-input path (its own stream)."""
    g = _gen(cfg.seed, 4, device)
    return torch.randn(cfg.T, cfg.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_expert(cfg: Config, e: int, device="cpu"):
    """(w1 [2I,...], w1_sf, w2 [H,...], w2_sf) for one expert."""
    g = _gen(cfg.seed, 1000 + e, device)
    w1 = torch.randn(2 * cfg.I, cfg.H, generator=g, device=device, dtype=torch.float32) * 0.02
    w2 = torch.randn(cfg.H, cfg.I, generator=g, device=device, dtype=torch.float32) * 0.02
    if cfg.variant == "mx":
        return quant_e2m1_ue8m0(w1) + quant_e2m1_ue8m0(w2)
    return quant_e4m3_f32_blocks(w1) + quant_e4m3_f32_blocks(w2)


def weight_shapes(cfg: Config):
    E, H, I = cfg.E + cfg.S, cfg.H, cfg.I
    if cfg.variant == "mx":
        return {"w1": ((E, 2 * I, H // 2), torch.uint8), "w1_sf": ((E, 2 * I, H // 32), torch.uint8),
                "w2": ((E, H, I // 2), torch.uint8), "w2_sf": ((E, H, I // 32), torch.uint8)}
    return {"w1": ((E, 2 * I, H), torch.uint8), "w1_sf": ((E, 2 * I // 128, H // 128), torch.float32),
            "w2": ((E, H, I), torch.uint8), "w2_sf": ((E, H // 128, I // 128), torch.float32)}


def make_weights(cfg: Config, device="cpu", experts: Optional[list] = None):
    """Stacked weights [E + S, ...] (shared experts last); experts not listed in
    `experts` stay zero."""
    shp = weight_shapes(cfg)
    out = {k: torch.zeros(s, dtype=dt, device=device) for k, (s, dt) in shp.items()}
    for e in (range(cfg.E + cfg.S) if experts is None else experts):
        w1, s1, w2, s2 = make_expert(cfg, e, device)
        out["w1"][e].copy_(w1)
        out["w1_sf"][e].copy_(s1)
        out["w2"][e].copy_(w2)
        out["w2_sf"][e].copy_(s2)
    return out


def make_inputs(cfg: Config, device="cpu", with_weights=True):
    idx, w = make_routing(cfg, device)
    x, x_sf = make_x(cfg, device)
    d = {"x": x, "x_sf": x_sf, "topk_idx": idx, "topk_w": w}
    if with_weights:
        d.update(make_weights(cfg, device))
    return d


def eval_rows(cfg: Config):
    """Rows the oracle evaluates: all tokens for the small configs, a seeded 1/64
    subset (sorted) for the large ones."""
    if cfg.T <= 256:
        return np.arange(cfg.T)
    rng = np.random.default_rng(cfg.seed + 7)
    return np.sort(rng.choice(cfg.T, cfg.T // 64, replace=False))


def to_numpy(d):
    return {k: (v.detach().cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
