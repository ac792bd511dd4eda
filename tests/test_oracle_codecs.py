"""Pins for the oracle's number formats (bf16 and FP8 E4M3).

bf16 is pinned to the rounding formula and the worked cancellation case in
"Deep Dive - DeepEP", "Combine: reverse routing plus reduction", to an
exhaustive round trip, and to PyTorch's own float32 -> bfloat16 cast.  E4M3 is
pinned to the OCP format definition exhaustively (every code, every midpoint)
and to PyTorch's float8_e4m3fn cast inside the finite range.
"""

import math
import struct

import numpy as np
import pytest
import torch

import oracle


def f32_bits(v):
    return struct.unpack("<I", struct.pack("<f", v))[0]


def bits_f32(u):
    return struct.unpack("<f", struct.pack("<I", u))[0]


# ----------------------------------------------------------------- bf16 -----

def test_bf16_page_cancellation_case(golden):
    g = dict(golden("worked_values.txt"))
    terms = [float(v) for v in g["p9_terms"]]
    # one final cast of the fp32 sum
    single = oracle.bf16_to_f32(oracle.f32_to_bf16(np.float32(terms[0] + terms[1] + terms[2])))
    assert single == float(g["p9_single_stage"][0])
    # a bf16 subtotal of the first two terms
    local = oracle.bf16_to_f32(oracle.f32_to_bf16(np.float32(terms[0] + terms[1])))
    assert local == float(g["p9_local_subtotal"][0])
    two = oracle.bf16_to_f32(oracle.f32_to_bf16(np.float32(local + terms[2])))
    assert two == float(g["p9_two_stages"][0])


def test_bf16_exhaustive_roundtrip():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f32_array(h)
    back = oracle.f32_to_bf16_array(f)
    nan = np.isnan(f)
    assert np.array_equal(back[~nan], h[~nan])
    # NaNs come back as quiet NaNs of the same sign
    assert np.all((back[nan] & 0x7FC0) == 0x7FC0)
    assert np.array_equal(back[nan] & 0x8000, h[nan] & 0x8000)


def test_bf16_matches_torch_cast():
    rng = np.random.default_rng(1)
    # random bit patterns over the whole finite range plus exact midpoints
    u = rng.integers(0, 2**32, 400000, dtype=np.uint64).astype(np.uint32)
    mids = (rng.integers(0, 2**16, 100000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    u = np.concatenate([u, mids, mids + 1, mids - 1]).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ours = oracle.f32_to_bf16_array(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_ties_to_even_examples():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even (1.0)
    assert oracle.f32_to_bf16(1.0 + 2.0**-8) == 0x3F80
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: to 1 + 2^-6
    assert oracle.f32_to_bf16(1.0 + 3 * 2.0**-8) == 0x3F82
    assert oracle.f32_to_bf16(-0.0) == 0x8000
    assert oracle.f32_to_bf16(float("inf")) == 0x7F80
    assert oracle.f32_to_bf16(bits_f32(0x7F7FFFFF)) == 0x7F80  # overflow


# ----------------------------------------------------------------- E4M3 -----

def _e4m3_values():
    codes = np.arange(256, dtype=np.uint8)
    return codes, oracle.e4m3_to_f32_array(codes)


def test_e4m3_decode_definition():
    codes, vals = _e4m3_values()
    assert vals[0x7E] == 448.0 and vals[0xFE] == -448.0
    assert math.isnan(vals[0x7F]) and math.isnan(vals[0xFF])
    assert vals[0x01] == 2.0**-9 and vals[0x08] == 2.0**-6
    assert vals[0x38] == 1.0 and vals[0x00] == 0.0
    assert math.copysign(1, vals[0x80]) < 0
    # positive finite codes are strictly increasing
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0)


def test_e4m3_exhaustive_roundtrip():
    codes, vals = _e4m3_values()
    back = oracle.f32_to_e4m3_array(vals)
    assert np.array_equal(back, codes)  # NaN -> NaN code of its sign too


def test_e4m3_midpoints_round_to_even():
    codes, vals = _e4m3_values()
    for sign in (1.0, -1.0):
        for c in range(0, 0x7E):
            lo, hi = float(vals[c]), float(vals[c + 1])
            mid = np.float32((lo + hi) / 2)
            assert float(mid) == (lo + hi) / 2  # exact in fp32
            even = c if c % 2 == 0 else c + 1
            got = oracle.f32_to_e4m3(sign * mid)
            assert got & 0x7F == even, (c, lo, hi)
            below = np.nextafter(mid, np.float32(0))
            above = np.nextafter(mid, np.float32(np.inf))
            assert oracle.f32_to_e4m3(sign * below) & 0x7F == c
            assert oracle.f32_to_e4m3(sign * above) & 0x7F == c + 1


def test_e4m3_satfinite_and_zero():
    assert oracle.f32_to_e4m3(448.0) == 0x7E
    assert oracle.f32_to_e4m3(463.99) == 0x7E
    assert oracle.f32_to_e4m3(464.0) == 0x7E    # tie between 448 and 480: even
    assert oracle.f32_to_e4m3(470.0) == 0x7E    # would round to 480: saturate
    assert oracle.f32_to_e4m3(1e30) == 0x7E
    assert oracle.f32_to_e4m3(-1e30) == 0xFE
    assert oracle.f32_to_e4m3(float("inf")) == 0x7E
    assert oracle.f32_to_e4m3(0.0) == 0x00
    assert oracle.f32_to_e4m3(-0.0) == 0x80
    assert oracle.f32_to_e4m3(2.0**-10) == 0x00      # tie 0 / 2^-9: even
    assert oracle.f32_to_e4m3(-(2.0**-11)) == 0x80   # rounds to -0


def test_e4m3_matches_torch_cast_in_range():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(2)
    v = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 50,
        rng.uniform(-448, 448, 200000).astype(np.float32),
        (rng.standard_normal(100000) * 2.0**-7).astype(np.float32),
    ])
    v = v[np.abs(v) <= 448]
    ours = oracle.f32_to_e4m3_array(v)
    ref = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
