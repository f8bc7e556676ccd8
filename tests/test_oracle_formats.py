"""Pins of the oracle's rounding points against the format definitions and
library conversions (CPU only).

BF16 and E4M3 encoders are checked against torch's own dtype casts (a
library routine), against every E4M3 code and every midpoint between
neighbouring codes (round-to-nearest-even by enumeration), and the MXFP8
block rule against hand-worked blocks in tests/golden/mxfp8_blocks.txt.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp8_blocks.txt")


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, vals, scale, codes = [p.strip() for p in line.split("|")]
            block = np.zeros(32)
            if vals.startswith("all="):
                block[:] = float(vals[4:])
            else:
                v = [float(s) for s in vals.split()]
                block[: len(v)] = v
            cases.append((name, block, int(scale), [int(c, 16) for c in codes.split()]))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_mxfp8_golden_blocks(case):
    name, block, scale, codes = case
    q, s = O.mx_quantize(block[None, :])
    assert int(s[0, 0]) == scale
    assert [int(c) for c in q[0, : len(codes)]] == codes
    if name.startswith("all"):
        assert all(int(c) == codes[0] for c in q[0])
    else:
        assert all(int(c) == 0 for c in q[0, len(codes):])


def test_e4m3_decode_table_points():
    # OCP E4M3: 1.0 = 0x38, largest finite 448 = 0x7E, smallest normal 2^-6 =
    # 0x08, smallest subnormal 2^-9 = 0x01, NaN = 0x7F.
    assert O.e4m3_decode(0x38) == 1.0
    assert O.e4m3_decode(0x7E) == 448.0
    assert O.e4m3_decode(0x08) == 2.0 ** -6
    assert O.e4m3_decode(0x01) == 2.0 ** -9
    assert O.e4m3_decode(0xB8) == -1.0
    assert math.isnan(O.e4m3_decode(0x7F))


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = O.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(v)
        else:
            assert v == ref[c], hex(c)


def test_e4m3_every_code_roundtrips():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert O.e4m3_encode(O.e4m3_decode(c)) == c, hex(c)


def test_e4m3_midpoints_round_to_even():
    pos = sorted({O.e4m3_decode(c) for c in range(0x7F)})
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = 0.5 * (lo + hi)
        clo, chi = O.e4m3_encode(lo), O.e4m3_encode(hi)
        even = clo if clo % 2 == 0 else chi
        assert O.e4m3_encode(mid) == even, (lo, hi)
        assert O.e4m3_encode(-mid) == even | 0x80
        assert O.e4m3_encode(np.nextafter(mid, 0)) == clo
        assert O.e4m3_encode(np.nextafter(mid, 1e9)) == chi


def test_e4m3_saturates_and_keeps_sign_of_zero():
    assert O.e4m3_encode(448.0) == 0x7E
    assert O.e4m3_encode(1e30) == 0x7E
    assert O.e4m3_encode(-1e30) == 0xFE
    assert O.e4m3_encode(0.0) == 0x00
    assert O.e4m3_encode(-0.0) == 0x80
    assert O.e4m3_encode(-(2.0 ** -11)) == 0x80


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.1, 1, 10, 100)])
    v = v[np.abs(v) < 448].astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([O.e4m3_encode(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(ours, ref)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.standard_normal(50000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # fp32 subnormals
        np.clip(rng.standard_normal(2000) * 3e38, -3.4e38, 3.4e38).astype(np.float32),
    ])
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    ours = O.bf16_round(v.astype(np.float64))
    assert np.array_equal(ours, ref)
    bits = O.bf16_bits(ours)
    assert np.array_equal(bits, torch.from_numpy(v).to(torch.bfloat16).view(torch.int16)
                          .numpy().view(np.uint16))
    assert np.array_equal(O.bf16_values(bits), ref)


def test_bf16_round_ties_and_overflow():
    one = 1.0
    ulp = 2.0 ** -7
    assert O.bf16_round(one + ulp / 2) == one            # tie to even (mantissa 0)
    assert O.bf16_round(one + 1.5 * ulp) == one + 2 * ulp  # tie to even (mantissa 2)
    big = (2 - 2 ** -7) * 2.0 ** 127
    assert O.bf16_round(big) == big
    assert O.bf16_round(big + 2.0 ** 119 * 0.99) == big     # below max + half ulp
    assert O.bf16_round(big + 2.0 ** 119) == math.inf        # tie at the top rounds up to inf


def test_mx_scale_exponent_rule():
    assert O.mx_scale_exponent(1.0) == -8
    assert O.mx_scale_exponent(448.0) == 0
    assert O.mx_scale_exponent(511.9) == 0
    assert O.mx_scale_exponent(512.0) == 1
    assert O.mx_scale_exponent(0.0) == -127
    assert O.mx_scale_exponent(2.0 ** -130) == -127
    assert O.mx_scale_exponent(2.0 ** 127) == 119


def test_mx_block_error_bound_and_scale_range():
    rng = np.random.default_rng(11)
    a = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    q, s = O.mx_quantize(a)
    deq = O.mx_dequantize(q, s)
    for r in range(64):
        for b in range(8):
            blk = a[r, 32 * b: 32 * b + 32]
            x = int(s[r, b]) - 127
            amax = np.abs(blk).max()
            assert 2.0 ** (x + 8) <= amax < 2.0 ** (x + 9)
            # RNE on the E4M3 grid: error at most half an ulp of the element's
            # binade (relative 2^-4), or half the subnormal quantum 2^-10.
            err = np.abs(deq[r, 32 * b: 32 * b + 32] - blk)
            bound = np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** (x - 10))
            over = np.abs(blk) > 448 * 2.0 ** x
            assert np.all(err[~over] <= bound[~over] * (1 + 1e-12))
