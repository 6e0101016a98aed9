"""CPU oracle for the MegaMoE forward of one MoE layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference arm
use it.  It shares no code, table or helper with the CUDA library.

What it computes is the plain definition of the unfused five-kernel chain the
fused MegaMoE kernel is bit-equal to (llm-infra-atlas "07 · MegaMoE", §0 and §1:
dispatch -> grouped GEMM L1 -> swiglu_apply_weight_to_fp8 -> grouped GEMM L2 ->
combine), with every expert local:

  1. x_hat[h]   = dec(x[t,h]) * S_x                      (block-scaled activations)
  2. W_hat      = dec(w) * S_w                           (block-scaled weights)
  3. g_j, u_j   = W1_hat[j] . x_hat, W1_hat[I+j] . x_hat  (fp64; rows [0,I) gate,
                  [I,2I) up: MEGAMOE_SM90_DESIGN.md §15.1 weight transform)
  4. a_j        = silu(g_j) * u_j * w[t,k]               (scaled SwiGLU, the
                  router weight folded in: "07 · MegaMoE" §8; design doc §10.1)
  5. requantise a to e4m3 per block along I (UE8M0 per 32 for the MX format,
     "07 · MegaMoE" §8; raw fp32 amax/448 per 128 or per 64 for the FP8
     format, DeepGEMM PR #440 "Why the order and not the pool size" on the raw
     scale and "Ring sizing, recycling, and why that granularity" on the width)
  6. y_k[h]     = W2_hat[h] . a_hat                      (fp64)
  7. out[t,h]   = bf16_rne(sum_k y_k[h])                 (the combine is a plain
                  sum because the weight was applied in step 4: "07 · MegaMoE" §9)

Shared experts (optional, `shared` > 0): experts E .. E+shared-1, which every
token uses with weight 1 after its K routed slots; their outputs are slots
K .. K+shared-1 of the same fixed-order sum.  The pages leave shared experts
out of the fused kernel (PR #440 "What a per-rank token count changes": no
shared-expert fusion, as in #383); this is the plain reading of a shared expert
as a routed expert every token selects with weight 1.

Where floating point decides an integer (the requantised codes and their
scale), the decision is taken in fp32, the precision the pages' epilogues run in
(design doc §10.1 works on float registers): the fp64 activation is rounded to
fp32 first.  Everything else is fp64.

Routing (step a1) is the plain definition of the contiguous per-expert pool
("07 · MegaMoE" §4; nxmr.cn walkthrough §二.2.4): experts in index order, each
segment padded to a multiple of the block size, and inside a segment the
(token, slot) pairs in ascending order (a deterministic order, fixed here in
place of the pages' round-robin over source ranks).
"""
from __future__ import annotations

import math
from typing import Callable, Dict, Iterable, Optional, Tuple

import numpy as np

# ----------------------------------------------------------------------------- codecs


def _e4m3_values() -> np.ndarray:
    """All 256 e4m3 (fn) codes from the bit-field definition: 1 sign, 4 exponent
    (bias 7), 3 mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN."""
    out = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0:
            v = (m / 8.0) * 2.0 ** -6
        elif e == 15 and m == 7:
            v = math.nan
        else:
            v = (1.0 + m / 8.0) * 2.0 ** (e - 7)
        out[c] = sign * v
    return out


def _e2m1_values() -> np.ndarray:
    """All 16 e2m1 codes: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0
    is subnormal (0 or 0.5)."""
    out = np.empty(16, dtype=np.float64)
    for c in range(16):
        sign = -1.0 if c & 0x8 else 1.0
        e = (c >> 1) & 0x3
        m = c & 0x1
        v = (m * 0.5) if e == 0 else (1.0 + m * 0.5) * 2.0 ** (e - 1)
        out[c] = sign * v
    return out


E4M3 = _e4m3_values()
E2M1 = _e2m1_values()
_E4M3_POS = E4M3[:127].copy()          # codes 0x00..0x7E: finite, non-negative, ascending
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    return E4M3[np.asarray(codes, dtype=np.uint8)]


def e2m1_decode(nibbles) -> np.ndarray:
    return E2M1[np.asarray(nibbles, dtype=np.uint8) & 0xF]


def ue8m0_decode(b) -> np.ndarray:
    """UE8M0 byte b -> 2^(b-127)."""
    return np.ldexp(1.0, np.asarray(b, dtype=np.int64) - 127)


def e4m3_encode_rne(v) -> np.ndarray:
    """Round each (exactly given) value to the nearest e4m3 value, ties to the even
    code, saturating at +-448.  Negative inputs keep the sign bit (so -tiny -> 0x80)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS, a, side="left")          # first value >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS[hi] - a
    d_lo = a - _E4M3_POS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(d_hi == 0, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)


def bf16_rne(v) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value (8 significant bits,
    exponent range of fp32), ties to even; returned as fp64."""
    v = np.asarray(v, dtype=np.float64)
    _, ex = np.frexp(v)
    q = np.maximum(ex - 8, -133)                     # quantum exponent (subnormals: 2^-133)
    r = np.rint(np.ldexp(v, -q))                     # exact scaling; rint = half to even
    out = np.ldexp(r, q)
    return np.where(np.abs(out) > 3.3895313892515355e38, np.copysign(np.inf, v), out)


# ----------------------------------------------------------------------------- requantisation


def ue8m0_exponent(amax) -> np.ndarray:
    """Smallest integer e with 448 * 2^e >= max(amax, 1e-10) (amax given as fp32),
    clamped to [-127, 127].  Exact: 448 = 0.875 * 2^9, amax = m * 2^ex."""
    amax = np.maximum(np.asarray(amax, dtype=np.float32), np.float32(1e-10)).astype(np.float64)
    m, ex = np.frexp(amax)
    e = np.where(m <= 0.875, ex - 9, ex - 8)
    return np.clip(e, -127, 127).astype(np.int64)


def requant_mx(a32: np.ndarray, block: int = 32) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """a32 fp32 [n] -> (e4m3 codes u8 [n], UE8M0 bytes u8 [n/block], dequantised fp64 [n]).
    Per block: e = ue8m0_exponent(amax); code = RNE_e4m3(a * 2^-e)."""
    a32 = np.asarray(a32, dtype=np.float32)
    n = a32.shape[-1]
    blocks = a32.reshape(n // block, block)
    amax = np.abs(blocks).max(axis=1)
    e = ue8m0_exponent(amax)
    scaled = blocks.astype(np.float64) * np.ldexp(1.0, -e)[:, None]
    codes = e4m3_encode_rne(scaled)
    deq = e4m3_decode(codes) * np.ldexp(1.0, e)[:, None]
    return codes.reshape(n), (e + 127).astype(np.uint8), deq.reshape(n)


def requant_f8(a32: np.ndarray, block: int = 128) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """a32 fp32 [n] -> (e4m3 codes [n], fp32 scales [n/block], dequantised fp64 [n]).
    Per block: s = fp32(max(amax,1e-10) / 448); code = RNE_e4m3(fp32(a / s))."""
    a32 = np.asarray(a32, dtype=np.float32)
    n = a32.shape[-1]
    blocks = a32.reshape(n // block, block)
    amax = np.maximum(np.abs(blocks).max(axis=1), np.float32(1e-10))
    s = (amax / np.float32(448.0)).astype(np.float32)
    q = (blocks / s[:, None]).astype(np.float32)
    codes = e4m3_encode_rne(q)
    deq = e4m3_decode(codes) * s.astype(np.float64)[:, None]
    return codes.reshape(n), s, deq.reshape(n)


def f8_act_gran(H: int, I: int) -> int:
    """Width of the FP8 intermediate's scale blocks along I by the pages' shape rule
    (DeepGEMM PR #440, "Ring sizing, recycling, and why that granularity"): 128
    when H % 512 == 0 and 2 * I % 512 == 0, else 64."""
    return 128 if H % 512 == 0 and (2 * I) % 512 == 0 else 64


def quantise_x(x: np.ndarray, variant: str) -> Tuple[np.ndarray, np.ndarray]:
    """bf16 activations (given as their exact fp32 / fp64 values) [T, H] -> the
    layer's FP8 input: (e4m3 codes u8 [T, H], scales).  The pages feed the
    layer x already quantised ("07 · MegaMoE" §3: the buffer's input region
    holds x and x_sf) in the formats of step 5 above, so a bf16 row is
    quantised here with the same block rule: UE8M0 per 32 (requant_mx) for
    mx, fp32 amax/448 per 128 (requant_f8) for f8.  mx scales: UE8M0 bytes
    [T, H/32]; f8 scales: fp32 [T, H/128].  Blocks never straddle rows (H is
    a multiple of the block), so the whole matrix is one call."""
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    if variant == "mx":
        codes, sf, _ = requant_mx(x.reshape(T * H), 32)
        return codes.reshape(T, H), sf.reshape(T, H // 32)
    codes, sf, _ = requant_f8(x.reshape(T * H), 128)
    return codes.reshape(T, H), sf.reshape(T, H // 128)


# ----------------------------------------------------------------------------- dequantisation


def dequant_x(x_row: np.ndarray, sf_row: np.ndarray, variant: str) -> np.ndarray:
    """One token's activations: e4m3 codes times UE8M0 per 32 (mx) or fp32 per 128 (f8)."""
    vals = e4m3_decode(x_row)
    if variant == "mx":
        return vals * np.repeat(ue8m0_decode(sf_row), 32)
    return vals * np.repeat(np.asarray(sf_row, dtype=np.float64), 128)


def dequant_weight(w: np.ndarray, sf: np.ndarray, variant: str) -> np.ndarray:
    """One expert's [N, Kdim] weight.  mx: w packed e2m1 [N, Kdim/2] (low nibble =
    even column), sf UE8M0 [N, Kdim/32].  f8: w e4m3 [N, Kdim], sf fp32 [N/128, Kdim/128]."""
    if variant == "mx":
        w = np.asarray(w, dtype=np.uint8)
        N = w.shape[0]
        nib = np.empty((N, w.shape[1] * 2), dtype=np.uint8)
        nib[:, 0::2] = w & 0xF
        nib[:, 1::2] = w >> 4
        return e2m1_decode(nib) * np.repeat(ue8m0_decode(sf), 32, axis=1)
    vals = e4m3_decode(w)
    s = np.repeat(np.repeat(np.asarray(sf, dtype=np.float64), 128, axis=0), 128, axis=1)
    return vals * s


# ----------------------------------------------------------------------------- routing (a1)


def route(topk_idx: np.ndarray, E: int, block: int) -> Dict[str, np.ndarray]:
    """Contiguous per-expert pool.  cnt[e] = #{(t,k): idx[t,k] = e};
    blk_off[e] = sum_{e'<e} ceil(cnt[e']/block); slot[t,k] = blk_off[e]*block +
    rank of (t,k) among expert e's pairs in ascending (t,k); src[row] = t*K+k or -1.
    Indices outside [0, E) are masked (slot -1); `bad` counts those >= E or < -1."""
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, K = idx.shape
    valid = (idx >= 0) & (idx < E)
    bad = int(np.count_nonzero((idx >= E) | (idx < -1)))
    cnt = np.zeros(E, dtype=np.int64)
    for e in idx[valid]:
        cnt[e] += 1
    nblk = (cnt + block - 1) // block
    blk_off = np.concatenate([[0], np.cumsum(nblk)])
    slot = np.full((T, K), -1, dtype=np.int64)
    fill = np.zeros(E, dtype=np.int64)
    for t in range(T):                     # ascending (t, k): the deterministic order
        for k in range(K):
            if valid[t, k]:
                e = idx[t, k]
                slot[t, k] = blk_off[e] * block + fill[e]
                fill[e] += 1
    src = np.full(int(blk_off[-1]) * block, -1, dtype=np.int64)
    for t in range(T):
        for k in range(K):
            if slot[t, k] >= 0:
                src[slot[t, k]] = t * K + k
    return {"cnt": cnt, "blk_off": blk_off, "slot": slot, "src": src, "bad": bad}


# ----------------------------------------------------------------------------- forward


ExpertFn = Callable[[int], Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]]


def expert_from_arrays(w1, w1_sf, w2, w2_sf) -> ExpertFn:
    """Adapter: stacked [E, ...] arrays -> per-expert accessor."""
    return lambda e: (w1[e], w1_sf[e], w2[e], w2_sf[e])


def forward_pair(x_hat: np.ndarray, w: float, W1: np.ndarray, W2: np.ndarray, I: int,
                 variant: str, clamp: Optional[float] = None, f8_gran: int = 128):
    """Steps 3-6 for one (token, expert) pair.  Returns (y fp64 [H], codes, sf, a fp64).

    clamp: the optional activation clamp of "MEGAMOE_SM90_DESIGN.md" §10 (L1
    epilogue: SwiGLU + FP8 quantization): gate and up are each limited to
    [-clamp, clamp] before the SwiGLU.
    f8_gran: the FP8 format's requant block along I, 128 or 64 (PR #440's
    l2_act_sf_gran_k); with 64 the L2 contraction dequantises each 64-wide half
    of a 128-K step with its own scale ("MEGAMOE_SM90_DESIGN.md" §5.4)."""
    g = W1[:I] @ x_hat
    u = W1[I:] @ x_hat
    if clamp is not None:
        g = np.clip(g, -clamp, clamp)
        u = np.clip(u, -clamp, clamp)
    with np.errstate(over="ignore"):
        a = g / (1.0 + np.exp(-g)) * u * float(np.float32(w))
    a32 = a.astype(np.float32)
    if variant == "mx":
        codes, sf, a_hat = requant_mx(a32, 32)
    else:
        codes, sf, a_hat = requant_f8(a32, f8_gran)
    y = W2 @ a_hat
    return y, codes, sf, a


def forward(rows: Iterable[int], x: np.ndarray, x_sf: np.ndarray, topk_idx: np.ndarray,
            topk_w: np.ndarray, experts: ExpertFn, H: int, I: int, E: int, variant: str,
            keep_intermediate: bool = False, partials_bf16: bool = False, clamp: Optional[float] = None,
            f8_gran: int = 128, shared: int = 0):
    """Output rows out[t, :] (bf16 values as fp64) for the tokens in `rows`.

    Each (token, slot) pair is computed independently (forward_pair); the pairs
    are visited expert by expert only so that each expert is decoded once, which
    does not change any value.  Returns (out [len(rows), H], inter) where inter
    maps (t, k) -> (codes, sf) of the requantised intermediate when asked.

    partials_bf16: the combine of the pages' own design ("MEGAMOE_SM90_DESIGN.md"
    §11, L2 BF16 epilogue + combine): every per-slot output y_k is cast to bf16
    (round to nearest even) before the top-k sum, which then runs in fixed k order
    and is cast to bf16 once more.  Read here as bf16_rne of the fp64 y_k.

    f8_gran: the FP8 intermediate's scale width, 128 or 64 (f8_act_gran gives the pages' shape rule).
    shared: shared experts E .. E+shared-1 (`experts` serves them too), used by
    every token with weight 1 as slots K .. K+shared-1."""
    rows = [int(t) for t in rows]
    K = topk_idx.shape[1]
    gran = int(f8_gran)
    pairs: Dict[int, list] = {}
    for t in rows:
        for k in range(K):
            e = int(topk_idx[t, k])
            if 0 <= e < E:
                pairs.setdefault(e, []).append((t, k, float(topk_w[t, k])))
        for j in range(shared):
            pairs.setdefault(E + j, []).append((t, K + j, 1.0))
    x_hat = {t: dequant_x(x[t], x_sf[t], variant) for t in rows}
    y = {}
    inter = {}
    for e in sorted(pairs):
        w1, w1_sf, w2, w2_sf = experts(e)
        W1 = dequant_weight(w1, w1_sf, variant)
        W2 = dequant_weight(w2, w2_sf, variant)
        for (t, k, w) in pairs[e]:
            yk, codes, sf, _ = forward_pair(x_hat[t], w, W1, W2, I, variant, clamp, gran)
            y[(t, k)] = yk
            if keep_intermediate:
                inter[(t, k)] = (codes, sf)
    out = np.zeros((len(rows), H), dtype=np.float64)
    for i, t in enumerate(rows):
        acc = np.zeros(H, dtype=np.float64)
        for k in range(K + shared):                  # fixed slot order, shared experts last
            if (t, k) in y:
                acc = acc + (bf16_rne(y[(t, k)]) if partials_bf16 else y[(t, k)])
        out[i] = bf16_rne(acc)
    return out, inter
