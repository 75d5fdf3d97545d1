"""Pins of the oracle's own bf16 and e4m3 codecs (CPU only).

The codecs are written from the format definitions (bf16: upper half of an
IEEE-754 binary32, round to nearest even; OCP FP8 E4M3 "fn": bias 7, no
infinities, largest finite 448). They are pinned here against PyTorch's CPU
casts (library routines), exhaustive enumeration, and values that follow from
the definitions by hand.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- bf16 --------------------------------------------------------------------

def test_bf16_decode_all_patterns_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_decode(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_roundtrip_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    back = O.bf16_encode(O.bf16_decode(bits))
    nan = np.isnan(O.bf16_decode(bits))
    assert np.array_equal(back[~nan], bits[~nan])
    assert np.all(np.isnan(O.bf16_decode(back[nan])))


def test_bf16_encode_matches_torch_random_and_ties():
    rng = np.random.default_rng(7)
    u = rng.integers(0, 2**32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    # exact halfway cases, with odd and even kept halves
    half = (rng.integers(0, 2**16, size=20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    u = np.concatenate([u, half, np.array([0x3F808000, 0x3F818000, 0x7F7F8000, 0xFF7FFFFF, 0x00008000], np.uint32)])
    f = u.view(np.float32)
    keep = ~np.isnan(f)
    f = f[keep]
    ours = O.bf16_encode(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_hand_values():
    # 1 + 2^-8 is exactly half way between 1 and 1 + 2^-7: ties to even -> 1.0
    f = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 65280.0 + 128.0], dtype=np.float32)
    assert O.bf16_encode(f).tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x4780]


# ---- e4m3 --------------------------------------------------------------------

def _torch_e4m3_decode(codes):
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()


def test_e4m3_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    ours = O.e4m3_decode(codes)
    ref = _torch_e4m3_decode(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_format_values_by_hand():
    """Values fixed by the format definition (OCP 8-bit FP, E4M3)."""
    with open(os.path.join(GOLDEN, "e4m3_format_points.json")) as fh:
        g = json.load(fh)
    codes = np.array([int(c, 16) for c in g["codes"]], dtype=np.uint8)
    vals = np.array(g["values"], dtype=np.float32)
    assert np.array_equal(O.e4m3_decode(codes), vals)
    assert np.array_equal(O.e4m3_encode(vals), codes)


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)


def test_e4m3_midpoints_round_to_even():
    mags = O.e4m3_decode(np.arange(127, dtype=np.uint8)).astype(np.float64)
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (mags[:-1] + mags[1:]) / 2)  # exact in fp32
    got = O.e4m3_encode(mids)
    lo = np.arange(126)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(O.e4m3_encode(-mids), want | 0x80)
    # just above / below a midpoint goes to the nearer neighbour
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    assert np.array_equal(O.e4m3_encode(up), (lo + 1).astype(np.uint8))
    assert np.array_equal(O.e4m3_encode(dn), lo.astype(np.uint8))


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.uniform(-448, 448, 500_000),
        rng.standard_normal(300_000) * 2.0 ** rng.integers(-12, 8, 300_000),
    ]).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ours = O.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_all_bf16_values_scaled_into_range_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = O.bf16_decode(bits)
    f = f[np.isfinite(f) & (np.abs(f) <= 448)]
    ours = O.e4m3_encode(f)
    ref = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_to_largest_finite():
    v = np.array([448.0, 449.0, 463.9, 464.0, 1e6, np.inf, -500.0, -np.inf], dtype=np.float32)
    assert O.e4m3_encode(v).tolist() == [0x7E] * 6 + [0xFE] * 2
    assert O.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
