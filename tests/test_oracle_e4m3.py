"""Pins for the oracle's e4m3 codec (the format of the FP8 KV cache in
"Smaller, faster, safer: running Kimi and GLM at scale", section "Quantizing
the KV cache").  The codec is checked against things other than itself: the
OFP8 specification's printed table, torch's float8_e4m3fn cast (a library
routine), exact midpoints, and saturation by definition of "satfinite".
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ofp8_e4m3_table.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, bits, value = line.split()
        if bits == "-":
            continue
        code = int(bits.replace(".", ""), 2)
        rows.append((name, code, float(value)))
    return rows


def test_golden_spec_table_decode():
    rows = _golden_rows()
    assert len(rows) == 8
    for name, code, value in rows:
        got = oracle.e4m3_decode(code)
        if math.isnan(value):
            assert math.isnan(got), name
        else:
            assert got == value and math.copysign(1, got) == math.copysign(1, value), name


def test_decode_all_256_vs_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got) and c in (0x7F, 0xFF)
        else:
            assert got == ref[c], hex(c)
            assert math.copysign(1, got) == math.copysign(1, ref[c])


def test_every_finite_code_round_trips():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = oracle.e4m3_decode(c)
        assert oracle.e4m3_encode(v) == c, hex(c)


def _finite_positive_values():
    return [(c, oracle.e4m3_decode(c)) for c in range(0x00, 0x7F)]


def test_midpoints_round_to_even_and_neighbours_to_nearest():
    vals = _finite_positive_values()
    for (c0, v0), (c1, v1) in zip(vals[:-1], vals[1:]):
        mid = (v0 + v1) / 2.0
        assert float(np.float32(mid)) == mid  # midpoints are exact in fp32
        even = c0 if (c0 & 1) == 0 else c1
        assert oracle.e4m3_encode(mid) == even, (hex(c0), hex(c1))
        assert oracle.e4m3_encode(-mid) == even | 0x80
        below = float(np.nextafter(np.float32(mid), np.float32(0)))
        above = float(np.nextafter(np.float32(mid), np.float32(np.inf)))
        assert oracle.e4m3_encode(below) == c0
        assert oracle.e4m3_encode(above) == c1


def test_saturation_and_specials():
    for x in [448.0, 449.0, 463.99, 464.0, 480.0, 1e4, 3.4e38, float("inf")]:
        assert oracle.e4m3_encode(x) == 0x7E, x
        assert oracle.e4m3_encode(-x) == 0xFE, x
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F
    # smallest fp32 subnormal rounds to a signed zero
    tiny = float(np.float32(1.4e-45))
    assert oracle.e4m3_encode(tiny) == 0x00
    assert oracle.e4m3_encode(-tiny) == 0x80


def test_encode_vs_torch_cast_random():
    rng = np.random.default_rng(1234)
    parts = [
        rng.uniform(-448, 448, 200_000),
        rng.standard_normal(200_000) * 0.01,          # subnormal region of e4m3
        rng.standard_normal(200_000) * 30.0,
        np.exp(rng.uniform(-30, math.log(448.0), 200_000)) * rng.choice([-1, 1], 200_000),
    ]
    x = np.concatenate(parts).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_array(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_encode_bits_range_matches_scalar():
    first = 0x3F800000  # 1.0f
    out = oracle.e4m3_encode_bits_range(first, 4096)
    for i in range(0, 4096, 97):
        v = np.array([first + i], dtype=np.uint32).view(np.float32)[0]
        assert out[i] == oracle.e4m3_encode(float(v))


def test_scale_from_amax():
    for a in [1.0, 3.0, 4.0, 17.5, 1e-3, 65504.0]:
        assert oracle.scale_from_amax(a) == float(np.float32(a) / np.float32(448.0))
    assert oracle.scale_from_amax(0.0) == 1.0
    # an amax whose quotient underflows to zero also gets 1.0
    assert oracle.scale_from_amax(float(np.float32(1.4e-45))) == 1.0


@pytest.mark.parametrize("seed", [0, 1])
def test_quantisation_error_bound(seed):
    """|dec(enc(x/s))*s - x| <= 2^-4 |x| when |x/s| is in the normal range,
    else <= s * 2^-10 (half a subnormal step): the e4m3 grid spacing."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(50_000) * rng.uniform(0.1, 8)).astype(np.float32)
    amax = float(np.abs(x).max())
    s = np.float32(oracle.scale_from_amax(amax))
    q = (x / s).astype(np.float32)
    codes = oracle.e4m3_encode_array(q)
    deq = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * float(s)
    err = np.abs(deq - x.astype(np.float64))
    normal = np.abs(q) >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]) * (1 + 1e-6))
    assert np.all(err[~normal] <= float(s) * 2.0 ** -10 * (1 + 1e-6))
