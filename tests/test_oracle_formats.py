"""Pins of the oracle's number formats (MXFP4 weights, MXFP8 activations, fp8
shared-expert weights) against the format definitions, torch's independent
float8 codec and closed forms.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tests import _brute
from workloads import generate as gen


def test_e2m1_all_codes_match_golden():
    gold = _brute.e2m1_table()
    for c in range(16):
        v = orc.e2m1_value(c)
        assert v == gold[c]
        assert math.copysign(1, v) == math.copysign(1, gold[c])


def test_e4m3_all_codes_match_torch_decoder():
    ref = _brute.e4m3_table()
    for c in range(256):
        v = orc.e4m3_value(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(v) and math.isnan(ref[c])
        else:
            assert v == ref[c], c
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x01) == 2.0 ** -9
    assert orc.e4m3_value(0x08) == 2.0 ** -6


def test_ue8m0_all_codes():
    for c in range(255):
        assert orc.ue8m0_value(c) == math.ldexp(1.0, c - 127)
    assert math.isnan(orc.ue8m0_value(255))


def test_e4m3_encode_roundtrip_every_finite_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert orc.e4m3_encode(orc.e4m3_value(c)) == c, hex(c)


def test_e4m3_encode_ties_go_to_even_mantissa():
    for c in range(0, 126):
        lo, hi = orc.e4m3_value(c), orc.e4m3_value(c + 1)
        mid = (lo + hi) / 2
        want = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == want
        assert orc.e4m3_encode(-mid) == want | 0x80


def test_e4m3_encode_saturates_and_keeps_sign():
    for y in (448.0, 449.0, 463.9, 464.0, 500.0, 511.99, 1e9):
        assert orc.e4m3_encode(y) == 0x7E
        assert orc.e4m3_encode(-y) == 0xFE
    assert orc.e4m3_encode(0.0) == 0x00
    assert orc.e4m3_encode(-0.0) == 0x80
    assert orc.e4m3_encode(-(2.0 ** -11)) == 0x80          # negative underflow keeps sign


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(7)
    y = np.concatenate([rng.uniform(-448, 448, 3000), rng.normal(0, 1, 3000),
                        rng.normal(0, 1e-2, 1000)]).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in y], np.uint8)
    assert (got == ref).all()


def test_mxfp8_closed_forms():
    q, s = orc.mxfp8_quantize(np.ones(32))
    assert s[0] == 127 - 8 and (q == 0x78).all()            # 1.0 / 2^-8 = 256 = 1.0 * 2^8
    v = np.zeros(32); v[0] = 3.0; v[1] = -3.0
    q, s = orc.mxfp8_quantize(v)
    assert s[0] == 127 + 1 - 8 and q[0] == 0x7C and q[1] == 0xFC and (q[2:] == 0).all()
    v = np.full(32, 255 / 128)                               # v / X = 510 -> saturates
    q, s = orc.mxfp8_quantize(v)
    assert s[0] == 119 and (q == 0x7E).all()
    v = np.zeros(32); v[5] = -0.0
    q, s = orc.mxfp8_quantize(v)
    assert s[0] == 0 and q[5] == 0x80 and q[4] == 0x00      # all-zero block
    q, s = orc.mxfp8_quantize(np.full(32, 2.0 ** -150))    # exponent clamps at -127
    assert s[0] == 0 and (q == orc.e4m3_encode(2.0 ** -23)).all()


def test_mxfp8_of_bf16_rows_matches_independent_quantiser():
    rng = np.random.default_rng(3)
    f = rng.standard_normal((8, 512)).astype(np.float32)
    f[0, :32] = 0.0
    f[1, 32:64] *= 1e-30
    f[2, 64:96] *= 1e30
    bits = gen.bf16_bits_from_f32(f)
    q, s = orc.quantize_bf16(bits)
    rq, rs = _brute.mxfp8(gen.bf16_bits_to_f32(bits).astype(np.float64))
    assert (q == rq).all() and (s == rs).all()
    # each dequantised value is the nearest e4m3 point of x / X (or +-448 when
    # x / X is beyond the largest finite value)
    x = gen.bf16_bits_to_f32(bits).astype(np.float64)
    X = np.ldexp(1.0, s.astype(np.int64) - 127).repeat(32, axis=1)
    y, yd = x / X, _brute.dq_mxfp8(q, s) / X
    mag = np.abs(y)
    step = np.where(mag < 2.0 ** -6, 2.0 ** -9,
                    np.ldexp(1.0, np.floor(np.log2(np.maximum(mag, 2.0 ** -6))).astype(np.int64) - 3))
    sat = mag > 448
    assert (np.abs(yd - y)[~sat] <= step[~sat] / 2).all()
    assert (np.abs(yd[sat]) == 448).all()


def test_generator_e2m1_ties_match_golden():
    rows = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "mx_rounding.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(tuple(map(float, line.split())))
    y = np.array([r[0] for r in rows], np.float32)
    idx = gen._e2m1_index(y)
    assert np.array_equal(gen._E2M1_MAG[idx], np.array([r[1] for r in rows], np.float32))


def test_generator_mxfp4_roundtrip_within_half_step():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((64, 256)) / 16).astype(np.float32)
    q, s = gen.encode_mxfp4_rows(w)
    d = np.array([[orc.e2m1_value(c) for c in row] for row in
                  np.stack([q & 15, q >> 4], -1).reshape(64, 256)])
    d *= np.repeat([[orc.ue8m0_value(c) for c in row] for row in s], 32, axis=1)
    # scale 2^(floor(log2 amax)-2): the largest element lands in [4, 8) before rounding
    amax = np.abs(w.reshape(64, 8, 32)).max(-1)
    X = np.array([[orc.ue8m0_value(c) for c in row] for row in s])
    assert ((amax / X >= 4) & (amax / X < 8)).all()
    step = np.where(np.abs(w) / X.repeat(32, 1) < 2, 0.5, np.where(np.abs(w) / X.repeat(32, 1) < 4, 1.0, 2.0))
    err = np.abs(d - w) / X.repeat(32, 1)
    sat = np.abs(w) / X.repeat(32, 1) > 6
    assert (err[~sat] <= step[~sat] / 2 + 1e-12).all()
    assert (np.abs(d[sat]) == 6 * X.repeat(32, 1)[sat]).all()


def test_generator_fp8_tiles_match_torch_cast():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((256, 256)) / 16).astype(np.float32)
    q, s = gen.encode_fp8_tiles(w)
    for i in range(2):
        for j in range(2):
            X = orc.ue8m0_value(int(s[i, j]))
            tile = w[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)].astype(np.float64) / X
            assert np.abs(tile).max() >= 256 and np.abs(tile).max() < 512
            ref = torch.from_numpy(np.clip(tile, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8)
            assert (q[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)] == ref.numpy()).all()


@pytest.mark.parametrize("val", [0.0, 1.0, -2.5, 3.140625])
def test_bf16_bits_roundtrip(val):
    b = gen.bf16_bits_from_f32(np.array([val], np.float32))
    assert gen.bf16_bits_to_f32(b)[0] == np.float32(val)
