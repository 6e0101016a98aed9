"""Pins for the oracle's forward: an independent dense brute force, closed forms,
zero cases, a dense-MLP special case and permutation equivariance (CPU only)."""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W

TINY_MX = W.CONFIGS["tiny"]
TINY_F8 = W.Config("tiny_f8", T=24, H=256, I=256, E=4, K=2, variant="f8", seed=11)


# ------------------------------------------------------------------ independent brute force
def _bits_e2m1(n: torch.Tensor) -> torch.Tensor:
    s = 1 - 2 * ((n >> 3) & 1).double()
    e = ((n >> 1) & 3).double()
    m = (n & 1).double()
    mag = torch.where(e == 0, 0.5 * m, (1 + 0.5 * m) * torch.exp2(e - 1))
    return s * mag


def _deq_all(cfg, inp):
    """Dense dequantised x [T,H], W1 [E,2I,H], W2 [E,H,I] in torch fp64."""
    x = inp["x"].view(torch.float8_e4m3fn).double()
    if cfg.variant == "mx":
        x = x * torch.exp2(inp["x_sf"].double() - 127).repeat_interleave(32, -1)
        def wq(p, sf):
            n = torch.stack([p & 0xF, p >> 4], -1).flatten(-2)
            return _bits_e2m1(n) * torch.exp2(sf.double() - 127).repeat_interleave(32, -1)
    else:
        x = x * inp["x_sf"].double().repeat_interleave(128, -1)
        def wq(c, sf):
            s = sf.double().repeat_interleave(128, -2).repeat_interleave(128, -1)
            return c.view(torch.float8_e4m3fn).double() * s
    return x, wq(inp["w1"], inp["w1_sf"]), wq(inp["w2"], inp["w2_sf"])


def _requant_torch(a32: torch.Tensor, variant: str, gran: int = 128) -> torch.Tensor:
    """Independent requant: library e4m3 cast, frexp-based exponent; FP8 blocks of `gran`."""
    n = a32.shape[-1]
    if variant == "mx":
        b = a32.reshape(*a32.shape[:-1], n // 32, 32)
        amax = b.abs().amax(-1).clamp_min(1e-10)
        m, ex = torch.frexp(amax)
        e = torch.where(m <= 0.875, ex - 9, ex - 8).clamp(-127, 127).double()
        q = (b.double() * torch.exp2(-e)[..., None]).float().to(torch.float8_e4m3fn)
        return (q.double() * torch.exp2(e)[..., None]).reshape(a32.shape)
    b = a32.reshape(*a32.shape[:-1], n // gran, gran)
    s = b.abs().amax(-1).clamp_min(1e-10) / 448.0
    q = (b / s[..., None]).to(torch.float8_e4m3fn)
    return (q.double() * s.double()[..., None]).reshape(a32.shape)


def brute_force(cfg, inp, partials_bf16=False, clamp=None, gran=128):
    """Dense per-slot loop; shared experts (cfg.S) as slots K .. K+S-1 that every
    token uses with weight 1."""
    x, W1, W2 = _deq_all(cfg, inp)
    T, I = cfg.T, cfg.I
    idx = torch.cat([inp["topk_idx"].long(), torch.arange(cfg.E, cfg.E + cfg.S).expand(T, cfg.S)], 1)
    w = torch.cat([inp["topk_w"].double(), torch.ones(T, cfg.S, dtype=torch.float64)], 1)
    out = torch.zeros(T, cfg.H, dtype=torch.float64)
    for k in range(cfg.K + cfg.S):
        valid = (idx[:, k] >= 0) & (idx[:, k] < cfg.E + cfg.S)
        e = idx[:, k].clamp(0, cfg.E + cfg.S - 1)
        h = torch.einsum("tnh,th->tn", W1[e], x)
        g, u = h[:, :I], h[:, I:]
        if clamp is not None:
            g, u = g.clamp(-clamp, clamp), u.clamp(-clamp, clamp)
        a = torch.nn.functional.silu(g) * u * w[:, k:k + 1]
        ah = _requant_torch(a.float(), cfg.variant, gran)
        y = torch.einsum("thi,ti->th", W2[e], ah)
        if partials_bf16:                  # library cast, round to nearest even
            y = y.to(torch.bfloat16).double()
        out += torch.where(valid[:, None], y, torch.zeros_like(y))
    return out


def run_oracle(cfg, inp, rows=None, partials_bf16=False, clamp=None, f8_gran=128):
    npi = W.to_numpy(inp)
    rows = np.arange(cfg.T) if rows is None else rows
    out, inter = O.forward(rows, npi["x"], npi["x_sf"], npi["topk_idx"], npi["topk_w"],
                           O.expert_from_arrays(npi["w1"], npi["w1_sf"], npi["w2"], npi["w2_sf"]),
                           cfg.H, cfg.I, cfg.E, cfg.variant, keep_intermediate=True, partials_bf16=partials_bf16,
                           clamp=clamp, f8_gran=f8_gran, shared=cfg.S)
    return out, inter


@pytest.mark.parametrize("cfg", [TINY_MX, TINY_F8, TINY_MX.with_(seed=5, K=3)], ids=["mx", "f8", "mx_k3"])
def test_oracle_matches_dense_brute_force(cfg):
    inp = W.make_inputs(cfg, "cpu")
    out, _ = run_oracle(cfg, inp)
    ref = O.bf16_rne(brute_force(cfg, inp).numpy())
    assert np.isfinite(out).all() and np.abs(out).max() > 0
    exact = np.mean(out == ref)
    assert exact > 0.999, exact
    assert np.max(np.abs(out - ref)) <= 2.0 ** -7 * np.max(np.abs(ref))


@pytest.mark.parametrize("cfg", [TINY_MX.with_(seed=5, K=3), TINY_F8], ids=["mx_k3", "f8"])
def test_oracle_bf16_partials_match_dense_brute_force(cfg):
    """The bf16-partials combine (each slot's output cast to bf16 before the sum)
    against the independent brute force with torch's bf16 cast."""
    inp = W.make_inputs(cfg, "cpu")
    out, _ = run_oracle(cfg, inp, partials_bf16=True)
    ref = O.bf16_rne(brute_force(cfg, inp, partials_bf16=True).numpy())
    assert np.mean(out == ref) > 0.999
    assert np.max(np.abs(out - ref)) <= 2.0 ** -7 * np.max(np.abs(ref))
    full, _ = run_oracle(cfg, inp)
    assert not np.array_equal(out, full)     # the extra rounding is visible with K > 1


@pytest.mark.parametrize("cfg", [TINY_MX.with_(seed=6, K=3), TINY_F8], ids=["mx_k3", "f8"])
def test_oracle_activation_clamp_matches_dense_brute_force(cfg):
    """Gate and up clamped to [-c, c] before the SwiGLU, with c small enough
    that most pre-activations are clamped; a huge c changes nothing."""
    inp = W.make_inputs(cfg, "cpu")
    out, _ = run_oracle(cfg, inp, clamp=0.05)
    ref = O.bf16_rne(brute_force(cfg, inp, clamp=0.05).numpy())
    assert np.mean(out == ref) > 0.999
    assert np.max(np.abs(out - ref)) <= 2.0 ** -7 * np.max(np.abs(ref))
    free, _ = run_oracle(cfg, inp)
    assert not np.array_equal(out, free)
    loose, _ = run_oracle(cfg, inp, clamp=1e30)
    assert np.array_equal(loose, free)


def test_oracle_bf16_partials_single_slot_equal_fp32_partials():
    """With one slot per token the sum has one term: bf16(bf16(y)) = bf16(y)."""
    cfg = TINY_MX.with_(K=1, seed=9)
    inp = W.make_inputs(cfg, "cpu")
    a, _ = run_oracle(cfg, inp, partials_bf16=True)
    b, _ = run_oracle(cfg, inp)
    assert np.array_equal(a, b)


def test_oracle_identity_weights_closed_form():
    """W1 gate = 2*[I|0], up = [I|0] and W2 = [I;0] (exact in e2m1 with UE8M0 scales):
    out[t, j<I] = bf16(sum_k deq(q(silu(2 x_j) * x_j * w_k))) and out[t, j>=I] = 0."""
    cfg = TINY_MX.with_(seed=3)
    inp = W.make_inputs(cfg, "cpu", with_weights=False)
    E, H, I = cfg.E, cfg.H, cfg.I
    eye = torch.zeros(I, H)
    eye[:, :I] = torch.eye(I)
    w1 = torch.cat([2.0 * eye, eye], 0)
    w2 = torch.zeros(H, I)
    w2[:I] = torch.eye(I)
    p1, s1 = W.quant_e2m1_ue8m0(w1)
    p2, s2 = W.quant_e2m1_ue8m0(w2)
    inp.update(w1=p1.expand(E, -1, -1).contiguous(), w1_sf=s1.expand(E, -1, -1).contiguous(),
               w2=p2.expand(E, -1, -1).contiguous(), w2_sf=s2.expand(E, -1, -1).contiguous())
    out, _ = run_oracle(cfg, inp)
    npi = W.to_numpy(inp)
    for t in range(cfg.T):
        xh = O.e4m3_decode(npi["x"][t]) * np.repeat(2.0 ** (npi["x_sf"][t].astype(int) - 127), 32)
        acc = np.zeros(H)
        for k in range(cfg.K):
            xj = xh[:I]
            a = (2 * xj) / (1 + np.exp(-2 * xj)) * xj * float(npi["topk_w"][t, k])
            _, _, ah = O.requant_mx(a.astype(np.float32), 32)
            acc[:I] += ah
        assert np.array_equal(out[t], O.bf16_rne(acc))
    assert np.all(out[:, I:] == 0)


@pytest.mark.parametrize("zero", ["x", "w", "w2"])
def test_oracle_zero_cases(zero):
    cfg = TINY_MX.with_(seed=4)
    inp = W.make_inputs(cfg, "cpu")
    if zero == "x":
        inp["x"].zero_()
    elif zero == "w":
        inp["topk_w"].zero_()
    else:
        inp["w2"].zero_()
    out, inter = run_oracle(cfg, inp)
    assert np.all(out == 0)


def test_oracle_dense_mlp_special_case():
    """E=1, K=1, w=1: a dense SwiGLU MLP with one requantisation of the hidden layer."""
    cfg = W.Config("mlp", T=16, H=256, I=128, E=1, K=1, seed=9)
    inp = W.make_inputs(cfg, "cpu")
    inp["topk_w"].fill_(1.0)
    out, _ = run_oracle(cfg, inp)
    x, W1, W2 = _deq_all(cfg, inp)
    h = x @ W1[0].T
    a = torch.nn.functional.silu(h[:, :cfg.I]) * h[:, cfg.I:]
    ref = _requant_torch(a.float(), "mx") @ W2[0].T
    assert np.mean(out == O.bf16_rne(ref.numpy())) > 0.999


def test_oracle_masked_slots_contribute_nothing():
    cfg = TINY_MX.with_(seed=6, K=2)
    inp = W.make_inputs(cfg, "cpu")
    base, _ = run_oracle(cfg, inp)
    inp2 = {k: v.clone() for k, v in inp.items()}
    inp2["topk_idx"][:, 1] = -1
    only0, _ = run_oracle(cfg, inp2)
    inp3 = {k: v.clone() for k, v in inp.items()}
    inp3["topk_idx"][:, 0] = -1
    only1, _ = run_oracle(cfg, inp3)
    assert not np.array_equal(base, only0)
    # removing a slot removes exactly its contribution (up to the final bf16 rounding)
    assert np.max(np.abs(O.bf16_rne(only0 + only1) - base)) <= 2.0 ** -6 * np.abs(base).max()
    inp2["topk_idx"][:, 0] = -1
    none, _ = run_oracle(cfg, inp2)
    assert np.all(none == 0)


def test_oracle_permutation_equivariance():
    cfg = TINY_MX.with_(seed=8)
    inp = W.make_inputs(cfg, "cpu")
    out, _ = run_oracle(cfg, inp)
    perm = torch.randperm(cfg.T, generator=torch.Generator().manual_seed(0))
    inp2 = dict(inp)
    for k in ("x", "x_sf", "topk_idx", "topk_w"):
        inp2[k] = inp[k][perm].contiguous()
    out2, _ = run_oracle(cfg, inp2)
    assert np.array_equal(out2, out[perm.numpy()])


def test_oracle_intermediate_codes_are_the_requant_of_the_activation():
    cfg = TINY_MX.with_(seed=12)
    inp = W.make_inputs(cfg, "cpu")
    _, inter = run_oracle(cfg, inp)
    x, W1, _ = _deq_all(cfg, inp)
    t, k = 5, 1
    e = int(inp["topk_idx"][t, k])
    h = W1[e] @ x[t]
    a = torch.nn.functional.silu(h[:cfg.I]) * h[cfg.I:] * float(inp["topk_w"][t, k])
    codes, sf = inter[(t, k)]
    assert np.array_equal(O.e4m3_decode(codes) * np.repeat(2.0 ** (sf.astype(int) - 127), 32),
                          _requant_torch(a.float()[None], "mx")[0].numpy())


# ------------------------------------------------------------------ FP8 intermediate scale width
def test_oracle_f8_gran_rule_on_the_pages_shapes():
    """DeepGEMM PR #440 runs its benchmark shapes (flash: H=4096, I=2048; pro:
    H=7168, I=3072) at the default width, 128; a hidden size or 2I that is not a
    multiple of 512 takes 64."""
    assert O.f8_act_gran(4096, 2048) == 128
    assert O.f8_act_gran(7168, 3072) == 128
    assert O.f8_act_gran(256, 256) == 64       # H % 512 != 0
    assert O.f8_act_gran(512, 128) == 64       # 2I = 256
    assert O.f8_act_gran(1024, 384) == 64      # 2I = 768
    assert O.f8_act_gran(1024, 256) == 128


@pytest.mark.parametrize("gran", [64, 128])
def test_oracle_f8_scale_width_matches_dense_brute_force(gran):
    """Per-64 and per-128 intermediate scales against the torch brute force; the
    two widths give different outputs on random data."""
    cfg = TINY_F8.with_(seed=13)
    inp = W.make_inputs(cfg, "cpu")
    out, inter = run_oracle(cfg, inp, f8_gran=gran)
    ref = O.bf16_rne(brute_force(cfg, inp, gran=gran).numpy())
    assert np.mean(out == ref) > 0.999
    assert np.max(np.abs(out - ref)) <= 2.0 ** -7 * np.max(np.abs(ref))
    codes, sf = next(iter(inter.values()))
    assert sf.shape == (cfg.I // gran,)
    other, _ = run_oracle(cfg, inp, f8_gran=192 - gran)
    assert not np.array_equal(out, other)


def test_oracle_f8_per64_equals_per128_when_halves_share_amax():
    """A 128-block whose two 64-halves have the same amax has the same scale and
    codes at either width (closed form of the raw-scale rule)."""
    rng = np.random.default_rng(4)
    a = rng.standard_normal(256).astype(np.float32)
    for b in range(2):                           # every half of both blocks peaks at +-3.5
        for h in range(2):
            seg = a[128 * b + 64 * h: 128 * b + 64 * h + 64]
            seg[np.argmax(np.abs(seg))] = np.float32(3.5) * np.sign(seg[np.argmax(np.abs(seg))])
    c64, s64, d64 = O.requant_f8(a, 64)
    c128, s128, d128 = O.requant_f8(a, 128)
    assert np.array_equal(c64, c128) and np.array_equal(d64, d128)
    assert np.array_equal(s64, np.repeat(s128, 2))


# ------------------------------------------------------------------ shared experts
SHARED = [TINY_MX.with_(seed=14, S=1), TINY_MX.with_(seed=15, S=2, K=3), TINY_F8.with_(seed=16, S=1)]


@pytest.mark.parametrize("cfg", SHARED, ids=["mx_s1", "mx_s2_k3", "f8_s1"])
def test_oracle_shared_experts_match_dense_brute_force(cfg):
    inp = W.make_inputs(cfg, "cpu")
    gran = 128 if cfg.variant == "mx" else O.f8_act_gran(cfg.H, cfg.I)
    out, inter = run_oracle(cfg, inp, f8_gran=gran)
    ref = O.bf16_rne(brute_force(cfg, inp, gran=gran).numpy())
    assert np.mean(out == ref) > 0.999
    assert np.max(np.abs(out - ref)) <= 2.0 ** -7 * np.max(np.abs(ref))
    assert all((t, cfg.K + j) in inter for t in range(cfg.T) for j in range(cfg.S))


def test_oracle_shared_expert_alone_is_a_dense_mlp():
    """Every routed slot masked: the output is the shared expert's SwiGLU MLP
    (weight 1) on every token."""
    cfg = TINY_MX.with_(seed=17, S=1)
    inp = W.make_inputs(cfg, "cpu")
    inp["topk_idx"].fill_(-1)
    out, _ = run_oracle(cfg, inp)
    x, W1, W2 = _deq_all(cfg, inp)
    h = x @ W1[cfg.E].T
    a = torch.nn.functional.silu(h[:, :cfg.I]) * h[:, cfg.I:]
    ref = _requant_torch(a.float(), "mx") @ W2[cfg.E].T
    assert np.mean(out == O.bf16_rne(ref.numpy())) > 0.999
    assert np.abs(out).max() > 0


def test_oracle_shared_expert_equals_a_routed_expert_every_token_picks():
    """The shared slot is the plain reading of a routed slot to expert E with weight
    1 appended to every token's routing."""
    cfg = TINY_MX.with_(seed=18, S=1)
    inp = W.make_inputs(cfg, "cpu")
    out, _ = run_oracle(cfg, inp)
    routed = cfg.with_(E=cfg.E + 1, K=cfg.K + 1, S=0)
    inp2 = dict(inp)
    inp2["topk_idx"] = torch.cat([inp["topk_idx"], torch.full((cfg.T, 1), cfg.E, dtype=torch.int32)], 1)
    inp2["topk_w"] = torch.cat([inp["topk_w"], torch.ones(cfg.T, 1)], 1)
    out2, _ = run_oracle(routed, inp2)
    assert np.array_equal(out, out2)
