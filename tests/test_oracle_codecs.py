"""Pins for the oracle's number formats and requantisation rules (CPU only)."""
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_decode_matches_library_for_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = O.e4m3_decode(np.arange(256))
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_e4m3_encode_matches_library_rne_on_grid_and_midpoints():
    pos = O.E4M3[:127]
    mids = (pos[:-1] + pos[1:]) / 2
    grid = np.concatenate([pos, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                           np.linspace(0, 448, 20011)])
    grid = np.concatenate([grid, -grid]).astype(np.float32)
    ref = torch.from_numpy(grid).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode_rne(grid.astype(np.float64))
    # compare by decoded value (+0 and -0 are the same number)
    assert np.array_equal(O.e4m3_decode(got), O.e4m3_decode(ref))


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if not math.isnan(O.E4M3[c])], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode_rne(O.e4m3_decode(codes)), codes)


def test_e4m3_saturates():
    assert O.e4m3_encode_rne(np.array([1e6]))[0] == 0x7E
    assert O.e4m3_encode_rne(np.array([-1e6]))[0] == 0xFE


def test_e2m1_values_closed_form():
    # e2m1 magnitudes: 0, the subnormal 0.5, and {1, 1.5} x 2^{0,1,2}
    mags = sorted({0.0, 0.5} | {m * 2.0 ** e for m in (1.0, 1.5) for e in (0, 1, 2)})
    assert list(O.E2M1[:8]) == mags
    assert list(O.E2M1[8:]) == [-m for m in mags]
    assert np.all(np.diff(O.E2M1[:8]) > 0)


def test_ue8m0_decode():
    assert O.ue8m0_decode(127) == 1.0
    assert O.ue8m0_decode(0) == 2.0 ** -127
    assert O.ue8m0_decode(254) == 2.0 ** 127


def test_bf16_rne_matches_library_on_fp32_inputs():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000),
                        [0.0, 1.0, -1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    got = O.bf16_rne(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rne_ties_to_even_exact_fp64():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1); 1 + 3*2^-8 -> 1 + 2^-6
    assert O.bf16_rne(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert O.bf16_rne(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    # just above the midpoint goes up: this needs fp64 input (not representable in fp32)
    assert O.bf16_rne(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 1 + 2.0 ** -7


def _golden_lines(prefix):
    with open(os.path.join(GOLDEN, "requant_blocks.txt")) as f:
        return [ln.split() for ln in f if ln.startswith(prefix + " ")]


@pytest.mark.parametrize("fields", _golden_lines("ue8m0"))
def test_ue8m0_rule_golden(fields):
    amax = struct.unpack("<f", struct.pack("<I", int(fields[1], 16)))[0]
    assert int(O.ue8m0_exponent(np.float32(amax))) == int(fields[2])


def _parse_block(line):
    txt = " ".join(line[1:])
    vals, scale, codes = [p.split() for p in txt.split("|")]
    return (np.array([float(v) for v in vals], dtype=np.float32), float(scale[1]),
            np.array([int(c, 16) for c in codes], dtype=np.uint8))


@pytest.mark.parametrize("line", _golden_lines("mxblock"))
def test_requant_mx_golden(line):
    vals, sf, codes = _parse_block(line)
    q, s, deq = O.requant_mx(vals, block=len(vals))
    assert int(s[0]) == int(sf)
    assert np.array_equal(O.e4m3_decode(q), O.e4m3_decode(codes))
    assert np.array_equal(deq, O.e4m3_decode(codes) * 2.0 ** (sf - 127))


@pytest.mark.parametrize("line", _golden_lines("f8block"))
def test_requant_f8_golden(line):
    vals, s_exp, codes = _parse_block(line)
    q, s, deq = O.requant_f8(vals, block=len(vals))
    assert float(s[0]) == s_exp
    assert np.array_equal(O.e4m3_decode(q), O.e4m3_decode(codes))


def test_requant_mx_scale_equivariance():
    # scaling a block by 2^j shifts its UE8M0 byte by j and keeps the codes
    rng = np.random.default_rng(1)
    a = (rng.standard_normal(64) * 3).astype(np.float32)
    q0, s0, d0 = O.requant_mx(a, 32)
    q1, s1, d1 = O.requant_mx((a * 2.0 ** 5).astype(np.float32), 32)
    assert np.array_equal(q0, q1) and np.array_equal(s1.astype(int) - s0.astype(int), [5, 5])
    assert np.array_equal(d1, d0 * 32)


def test_requant_mx_error_bound():
    # e4m3 has 3 mantissa bits: |a - deq| <= 2^-4 |a| for normals, plus 2^-10 * 2^e subnormal floor
    rng = np.random.default_rng(2)
    a = (rng.standard_normal(32 * 500) * np.repeat(10.0 ** rng.uniform(-8, 3, 500), 32)).astype(np.float32)
    q, s, d = O.requant_mx(a, 32)
    scale = np.repeat(2.0 ** (s.astype(np.int64) - 127), 32)
    err = np.abs(d - a.astype(np.float64))
    assert np.all(err <= np.abs(a) * 2.0 ** -4 + scale * 2.0 ** -10 + 0.0)
    blocks = np.abs(a).reshape(-1, 32).max(1)
    assert np.all(blocks <= 448 * 2.0 ** (s.astype(np.int64) - 127))
    assert np.all(blocks > 224 * 2.0 ** (s.astype(np.int64) - 127))   # smallest such e


@pytest.mark.parametrize("variant", ["mx", "f8"])
def test_quantise_x_matches_workload_quantiser(variant):
    """Two independent quantisers of the layer's FP8 input (the oracle's numpy
    requant and the input generator's torch one) agree bit for bit on bf16 rows."""
    import workload as W
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(37, 512, generator=g) * torch.logspace(-3, 3, 37)[:, None]).to(torch.bfloat16)
    codes, sf = O.quantise_x(x.float().numpy(), variant)
    if variant == "mx":
        rc, rs = W.quant_e4m3_ue8m0(x.float(), 32)
    else:
        rc, rs = W.quant_e4m3_f32_rows(x.float(), 128)
    assert np.array_equal(codes, rc.numpy())
    assert np.array_equal(np.asarray(sf), rs.numpy())


def test_quantise_x_closed_forms():
    """A row of ones: UE8M0 e = -8 (448 * 2^-8 = 1.75 >= 1 > 0.875), byte 119,
    every code 1 * 2^8 = 256 = 0x78; F8 s = fp32(1/448), code RNE(1/s) = 448 = 0x7E.
    A zero row: the 1e-10 floor, e = -42 (448 * 2^-42 >= 1e-10 > 448 * 2^-43), codes 0."""
    ones = np.ones((2, 256), dtype=np.float32)
    c, s = O.quantise_x(ones, "mx")
    assert np.all(s == 119) and np.all(c == 0x78)
    c, s = O.quantise_x(ones, "f8")
    assert np.all(s == np.float32(1.0) / np.float32(448.0)) and np.all(c == 0x7E)
    zero = np.zeros((1, 128), dtype=np.float32)
    c, s = O.quantise_x(zero, "mx")
    assert np.all(s == 127 - 42) and np.all(c == 0)
