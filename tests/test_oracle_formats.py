"""Pins for the oracle's storage-format codecs (bf16, fp16, e4m3fn).

Pinned against: the format specifications (golden landmark encodings), exhaustive round trips over
every code, ties-to-even at every midpoint, brute-force nearest-value search, and torch's own CPU
conversions (a library routine) on random values.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import GOLDEN

pytestmark = pytest.mark.filterwarnings("ignore")


def _parse_value(tok: str) -> float:
    if tok in ("nan", "inf", "-inf"):
        return float(tok)
    if "*2^" in tok:
        m, e = tok.split("*2^")
        return math.ldexp(float(m), int(e))
    return float(tok)


def _landmarks():
    rows = []
    with open(os.path.join(GOLDEN, "format_landmarks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, code, val = line.split()
            rows.append((fmt, int(code, 16), _parse_value(val), val))
    return rows


def _all_codes(fmt):
    if fmt == "e4m3":
        return torch.arange(256, dtype=torch.int32).to(torch.uint8)
    dt = torch.bfloat16 if fmt == "bf16" else torch.float16
    return torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(dt)


def _decode_code(orc, fmt, code):
    if fmt == "e4m3":
        return orc.decode(torch.tensor([code], dtype=torch.uint8)).item()
    dt = torch.bfloat16 if fmt == "bf16" else torch.float16
    c = torch.tensor([code if code < 32768 else code - 65536], dtype=torch.int16).view(dt)
    return orc.decode(c).item()


def _encode_value(orc, fmt, v):
    if fmt == "e4m3":
        return int(orc.encode(torch.tensor([v], dtype=torch.float32), "e4m3").item())
    dt = torch.bfloat16 if fmt == "bf16" else torch.float16
    return int(orc.encode(torch.tensor([v], dtype=torch.float32), dt).view(torch.int16).item()) & 0xFFFF


@pytest.mark.parametrize("row", _landmarks(), ids=lambda r: f"{r[0]}-{r[1]:x}")
def test_landmark_decode_and_encode(orc, row):
    fmt, code, value, text = row
    got = _decode_code(orc, fmt, code)
    if math.isnan(value):
        assert math.isnan(got)
        return
    assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value), (text, got)
    if math.isinf(value) or (fmt == "bf16" and value > 3.4e38):
        return
    assert _encode_value(orc, fmt, value) == code


@pytest.mark.parametrize("fmt", ["bf16", "fp16", "e4m3"])
def test_exhaustive_round_trip(orc, fmt):
    """decode then encode is the identity on every non-NaN code."""
    codes = _all_codes(fmt)
    vals = orc.decode(codes)
    nan = torch.isnan(vals)
    if fmt == "e4m3":
        assert int(nan.sum()) == 2  # only S.1111.111
        back = orc.encode(vals, "e4m3")
        assert torch.equal(back[~nan], codes[~nan])
    else:
        back = orc.encode(vals, codes.dtype)
        assert torch.equal(back.view(torch.int16)[~nan], codes.view(torch.int16)[~nan])


@pytest.mark.parametrize("fmt", ["bf16", "fp16", "e4m3"])
def test_exhaustive_decode_matches_torch(orc, fmt):
    codes = _all_codes(fmt)
    mine = orc.decode(codes)
    if fmt == "e4m3":
        ref = codes.view(torch.float8_e4m3fn).to(torch.float32)
    else:
        ref = codes.to(torch.float32)
    both_nan = torch.isnan(mine) & torch.isnan(ref)
    assert torch.equal(mine[~both_nan], ref[~both_nan])
    assert torch.equal(torch.isnan(mine), torch.isnan(ref))


def _positive_finite_sorted(orc, fmt):
    codes = _all_codes(fmt)
    vals = orc.decode(codes).double()
    keep = torch.isfinite(vals) & (vals >= 0) & ~((vals == 0) & (torch.signbit(vals)))
    v, idx = torch.sort(vals[keep])
    return v, codes[keep][idx]


@pytest.mark.parametrize("fmt", ["fp16", "e4m3"])
def test_every_midpoint_ties_to_even(orc, fmt):
    """The midpoint of two adjacent representable values rounds to the one with an even code."""
    v, codes = _positive_finite_sorted(orc, fmt)
    lo, hi = v[:-1], v[1:]
    mid = (lo + hi) / 2  # exact in fp64; also exact in fp32 for these formats
    mid32 = mid.to(torch.float32)
    assert torch.equal(mid32.double(), mid)
    if fmt == "e4m3":
        got = orc.encode(mid32, "e4m3").to(torch.int32)
        cl = codes[:-1].to(torch.int32)
        ch = codes[1:].to(torch.int32)
    else:
        got = orc.encode(mid32, torch.float16).view(torch.int16).to(torch.int32)
        cl = codes[:-1].view(torch.int16).to(torch.int32)
        ch = codes[1:].view(torch.int16).to(torch.int32)
    expect = torch.where(cl % 2 == 0, cl, ch)
    assert torch.equal(got, expect)


def test_bf16_midpoints_tie_to_even(orc):
    v, codes = _positive_finite_sorted(orc, "bf16")
    lo, hi = v[:-1], v[1:]
    mid = ((lo + hi) / 2).to(torch.float32)
    got = orc.encode(mid, torch.bfloat16).view(torch.int16).to(torch.int32)
    cl = codes[:-1].view(torch.int16).to(torch.int32)
    ch = codes[1:].view(torch.int16).to(torch.int32)
    assert torch.equal(got, torch.where(cl % 2 == 0, cl, ch))


def test_e4m3_brute_force_nearest(orc):
    """Each encoding is the nearest finite e4m3 value (brute force over all codes), ties to even."""
    rng = np.random.Generator(np.random.PCG64(7))
    mags = np.concatenate([rng.uniform(0, 448, 20000), np.exp(rng.uniform(np.log(1e-4), np.log(448), 20000))])
    vals = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    got = orc.encode(torch.from_numpy(vals), "e4m3")
    table_codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    table = orc.decode(table_codes).double().numpy()
    finite = np.isfinite(table)
    tv = table[finite]
    tc = np.arange(256)[finite]
    for v, c in zip(vals.astype(np.float64), got.numpy()):
        d = np.abs(tv - v)
        best = d.min()
        cands = tc[d == best]
        # prefer the candidate with an even mantissa (ties to even); +-0 are both fine for 0
        cands_even = [k for k in cands if k % 2 == 0] or list(cands)
        assert int(c) in cands_even or (best == 0 and int(c) in cands), (v, c, cands)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_encoder_matches_torch_random(orc, dt):
    """Encoding 1e6 random fp32 values (normal, subnormal and huge magnitudes) matches torch."""
    rng = np.random.Generator(np.random.PCG64(11))
    bits = rng.integers(0, 2**32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    vals = torch.from_numpy(bits.view(np.float32).copy())
    vals = vals[torch.isfinite(vals)]
    mine = orc.encode(vals, dt).view(torch.int16)
    ref = vals.to(dt).view(torch.int16)
    assert torch.equal(mine, ref)


def test_e4m3_encoder_matches_torch_random(orc):
    rng = np.random.Generator(np.random.PCG64(13))
    mags = np.exp(rng.uniform(np.log(1e-6), np.log(464.0), 1_000_000))
    vals = torch.from_numpy((mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32))
    vals = vals[vals.abs() <= 464.0]
    mine = orc.encode(vals, "e4m3")
    ref = vals.to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(mine, ref)


def test_e4m3_overflow_is_nan_not_inf(orc):
    """e4m3fn has no infinity: values that round past 448 encode as NaN (S.1111.111)."""
    vals = torch.tensor([464.0001, 480.0, 1e6, -500.0, float("inf")], dtype=torch.float32)
    got = orc.encode(vals, "e4m3")
    assert got.tolist() == [0x7F, 0x7F, 0x7F, 0xFF, 0x7F]
