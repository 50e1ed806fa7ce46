"""Pins for the oracle's e4m3 / bf16 / ue8m0 primitives (CPU only).

Each pin checks the oracle against something other than itself: the
float8_e4m3fn and bfloat16 casts of PyTorch (library routines), exact rational
arithmetic, and the closed-form properties of the format.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

TABLE = oracle.e4m3_decode_table()


def torch_e4m3_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_e4m3_encode(x):
    """Library cast with saturation applied first (the cast itself does not saturate)."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).clone()
    nan = torch.isnan(t)
    t = t.clamp(-448.0, 448.0)
    codes = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    codes[nan.numpy()] = 0x7F
    return codes


def test_decode_table_matches_library_cast():
    ref = torch_e4m3_decode_all()
    for c in range(256):
        if math.isnan(ref[c]):
            assert math.isnan(TABLE[c]), c
        else:
            assert TABLE[c] == ref[c], (c, TABLE[c], ref[c])
            assert math.copysign(1.0, TABLE[c]) == math.copysign(1.0, ref[c])


def test_decode_table_format_properties():
    nonneg = TABLE[:127]
    assert np.all(np.diff(nonneg) > 0), "non-negative codes must be strictly increasing"
    assert nonneg[0] == 0.0 and nonneg[1] == 2.0 ** -9 and nonneg[126] == 448.0
    assert math.isnan(TABLE[0x7F]) and math.isnan(TABLE[0xFF])
    assert np.isnan(TABLE).sum() == 2
    # sign symmetry
    for c in range(128):
        if c != 0x7F:
            assert TABLE[c | 0x80] == -TABLE[c]
    assert math.copysign(1.0, TABLE[0x80]) == -1.0


def test_round_trip_all_codes():
    vals = TABLE.astype(np.float32)
    enc = oracle.e4m3_encode(vals)
    for c in range(256):
        if c in (0x7F, 0xFF):
            assert enc[c] == 0x7F           # NaN encodes to the canonical NaN code
        else:
            assert enc[c] == c, (c, enc[c])


def midpoints():
    v = TABLE[:127]
    mids = (v[:-1] + v[1:]) / 2.0          # exact in fp64 and in fp32 (<= 5 significant bits)
    assert np.all(mids.astype(np.float32).astype(np.float64) == mids)
    return mids


def test_ties_go_to_even_code():
    mids = midpoints()
    enc = oracle.e4m3_encode(mids.astype(np.float32))
    for i, m in enumerate(mids):
        lo, hi = i, i + 1
        expect = lo if lo % 2 == 0 else hi
        assert enc[i] == expect, (m, enc[i], expect)
    encn = oracle.e4m3_encode((-mids).astype(np.float32))
    assert np.array_equal(encn, enc | 0x80)


def test_encode_matches_library_cast_dense():
    rng = np.random.default_rng(1234)
    mags = np.exp2(rng.uniform(-14.0, 10.0, size=400_000)).astype(np.float32)
    sgn = np.where(rng.random(mags.size) < 0.5, -1.0, 1.0).astype(np.float32)
    x = mags * sgn
    mids = midpoints().astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))])
    x = np.concatenate([x, near, -near, TABLE[:127].astype(np.float32)])
    assert np.array_equal(oracle.e4m3_encode(x), torch_e4m3_encode(x))


def test_saturation_and_specials():
    big = np.array([448.0, 448.5, 463.9, 464.0, 480.0, 1e4, 1e30, np.inf], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    assert oracle.e4m3_encode(np.array([np.nan], dtype=np.float32))[0] == 0x7F
    assert oracle.e4m3_encode(np.array([-0.0], dtype=np.float32))[0] == 0x80
    assert oracle.e4m3_encode(np.array([0.0], dtype=np.float32))[0] == 0x00
    # below half the smallest subnormal -> signed zero; exactly half -> tie to 0 (even)
    tiny = np.array([2.0 ** -11, 2.0 ** -10, -(2.0 ** -10), 2.0 ** -10 * 1.0000001], dtype=np.float32)
    assert list(oracle.e4m3_encode(tiny)) == [0x00, 0x00, 0x80, 0x01]


# --- bf16 rounding -----------------------------------------------------------

def bf16_bits_torch(x32):
    t = torch.from_numpy(np.asarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_value(bits):
    return float(np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0])


def bf16_nearest_bruteforce(x: Fraction) -> int:
    """Nearest bf16 to an exact rational, ties to even, by comparing candidates."""
    f = float(x)
    b = int(np.array([f], dtype=np.float32).view(np.uint32)[0] >> 16)
    cands = set()
    for d in (-2, -1, 0, 1, 2):
        c = (b + d) & 0xFFFF
        v = bf16_value(c)
        if math.isfinite(v):
            cands.add(c)
    best = None
    for c in sorted(cands):
        dist = abs(Fraction(bf16_value(c)) - x)
        key = (dist, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_bf16_from_fp32_matches_library():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(300_000) * np.exp2(rng.uniform(-30, 30, 300_000))).astype(np.float32)
    x = np.concatenate([x, np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, -1e-42], dtype=np.float32)])
    ours = oracle.bf16_rn(x.astype(np.float64))
    assert np.array_equal(ours, bf16_bits_torch(x))


def test_bf16_from_fp64_exact_rational():
    rng = np.random.default_rng(8)
    x = rng.standard_normal(3000) * np.exp2(rng.integers(-20, 20, 3000))
    # exact bf16 midpoints (ties) and values one fp64 ulp around them
    base = np.array([bf16_value(b) for b in rng.integers(0x3000, 0x4F00, 200)])
    ulp = np.array([bf16_value(int(np.array([v], np.float32).view(np.uint32)[0] >> 16) + 1) - v for v in base])
    mid = base + ulp / 2
    x = np.concatenate([x, mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf), -mid])
    ours = oracle.bf16_rn(x)
    for xi, oi in zip(x, ours):
        assert oi == bf16_nearest_bruteforce(Fraction(float(xi))), xi


# --- ue8m0 exponent rule -------------------------------------------------------

def ceil_log2_exact(r: Fraction) -> int:
    e = 0
    while Fraction(2) ** e < r:
        e += 1
    while Fraction(2) ** (e - 1) >= r:
        e -= 1
    return e


def test_ue8m0_exact_at_powers_of_two_of_448():
    # sglang pull request #43480, review item 7: groups placed on exact powers of two
    # of 448 must get exactly that power of two, one step up as soon as amax exceeds it.
    for k in range(-30, 31):
        amax = np.float32(448.0 * 2.0 ** k)
        assert oracle.ue8m0_byte(float(np.float32(amax / np.float32(448.0)))) == 127 + k
        above = np.nextafter(amax, np.float32(np.inf))
        assert oracle.ue8m0_byte(float(np.float32(above / np.float32(448.0)))) == 127 + k + 1


def test_ue8m0_matches_exact_ceil_log2():
    rng = np.random.default_rng(9)
    r = np.exp2(rng.uniform(-140, 100, 3000)).astype(np.float32)
    r = r[r > 0]
    for v in r:
        e = ceil_log2_exact(Fraction(float(v)))
        assert oracle.ue8m0_byte(float(v)) == max(0, min(254, e + 127)), v
    assert oracle.ue8m0_byte(0.0) == 0


def test_ue8m0_clamps_at_the_top_of_the_range():
    # ceil(log2 r) grows without bound as r does and the byte is clamped to 254: the largest
    # finite ratio (fp32 max / 448 ~ 2^119.2) still has its own exponent, and an infinite
    # ratio (a group holding an infinity) takes the clamp like any ratio above 2^127
    big = np.float32(np.finfo(np.float32).max / np.float32(448.0))
    assert oracle.ue8m0_byte(float(big)) == ceil_log2_exact(Fraction(float(big))) + 127
    assert oracle.ue8m0_byte(float(np.float32(2.0 ** 127))) == 254
    assert oracle.ue8m0_byte(float(np.nextafter(np.float32(2.0 ** 127), np.float32(np.inf)))) == 254
    assert oracle.ue8m0_byte(float("inf")) == 254
