"""Pins for the oracle's quantisers and the per-row fp8-wire codec (CPU only).

Checked against: the page's scale-granularity table (MORI GEMM + All-Reduce
Benchmark, 'What fp8 costs, numerically'), PyTorch's float8/bfloat16 casts
(library routines), and closed-form error bounds of the format.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic
from conftest import rel_l2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TABLE = oracle.e4m3_decode_table()


def dequant_block(codes, scales, gr, gc):
    R, C = codes.shape
    s = np.repeat(np.repeat(scales.astype(np.float64), gr, axis=0), gc, axis=1)[:R, :C]
    return TABLE[codes] * s


@pytest.fixture(scope="module")
def payload():
    # the page's payload: a [2048, 7168] standard-normal matrix
    return synthetic.normal(0, synthetic.TID_X, 0, (2048, 7168))


def test_scale_granularity_table(payload):
    with open(os.path.join(GOLDEN, "mori_fp8_cost_table.json")) as f:
        table = json.load(f)
    for row in table["rows"]:
        g = row["group"]
        codes, scales = oracle.quant_block(payload, 1, g)
        err = rel_l2(dequant_block(codes, scales, 1, g), payload)
        # a statistic of the distribution, printed to 4 digits: a 0.3% band around it
        assert abs(err - row["rel_l2"]) <= 0.003 * row["rel_l2"], (row["label"], err, row["rel_l2"])


def test_rowquant_matches_library_cast(payload):
    x = payload[:256]
    q, s = oracle.rowquant(x)
    t = torch.from_numpy(x)
    amax = t.abs().amax(dim=1)
    s_ref = amax / torch.tensor(448.0, dtype=torch.float32)
    assert np.array_equal(s, s_ref.numpy())
    q_ref = (t / s_ref[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, q_ref)
    # equals the generic block quantiser with one group per row
    q2, s2 = oracle.quant_block(x, 1, x.shape[1])
    assert np.array_equal(q, q2) and np.array_equal(s, s2[:, 0])


def test_rowdequant_matches_library_cast():
    rng = np.random.default_rng(3)
    q = rng.integers(0, 256, size=(64, 512), dtype=np.uint8)
    q[q == 0x7F] = 0x7E
    q[q == 0xFF] = 0xFE
    s = (rng.random(64) * 3).astype(np.float32)
    s[5] = 0.0
    y = oracle.rowdequant(q, s)
    qt = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float32)
    yref = (qt * torch.from_numpy(s)[:, None]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, yref)


def test_codec_zero_row_and_powers_of_two():
    x = np.zeros((4, 256), dtype=np.float32)
    x[1, :] = -0.0
    x[2, 7] = 448.0 * 8          # amax exactly 448*2^3: scale 8, that element encodes to 448
    x[2, 9] = -3.0
    x[3, :] = np.float32(2.0 ** -120)
    q, s = oracle.rowquant(x)
    assert s[0] == 0 and s[1] == 0 and np.all(q[:2] == 0)
    assert s[2] == 8.0 and q[2, 7] == 0x7E and TABLE[q[2, 9]] * 8 == -3.0
    y = oracle.rowdequant(q, s)
    assert np.all(y[:2] == 0)
    assert np.all(oracle.bf16_to_f32(y[3]) == np.float32(2.0 ** -120))


def test_codec_error_bound(payload):
    x = payload[:512]
    q, s = oracle.rowquant(x)
    deq = TABLE[q] * s[:, None].astype(np.float64)
    # e4m3 keeps 4 significant bits: relative half-spacing 2^-4 in the normal range,
    # absolute half-spacing 2^-10 * s in the subnormal range
    bound = np.abs(x) * 2.0 ** -4 + s[:, None] * 2.0 ** -10
    assert np.all(np.abs(deq - x) <= bound * (1 + 1e-12))
    # the largest element of every row lands on +-448 exactly
    amax_idx = np.abs(x).argmax(axis=1)
    assert np.all((q[np.arange(x.shape[0]), amax_idx] & 0x7F) == 0x7E)


def test_block_quant_128x128_properties():
    x = synthetic.normal(0, synthetic.TID_B, 0, (384, 512), sigma=0.02)
    x[128:256, 0:128] = 0.0                       # an all-zero block
    codes, scales = oracle.quant_weight_128x128(x)
    assert scales.shape == (3, 4)
    assert scales[1, 0] == 0 and np.all(codes[128:256, 0:128] == 0)
    for bi in range(3):
        for bj in range(4):
            blk = x[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            amax = np.abs(blk).max()
            assert scales[bi, bj] == np.float32(np.float32(amax) / np.float32(448.0))
            if amax > 0:
                c = codes[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
                assert (c.ravel()[np.abs(blk).argmax()] & 0x7F) == 0x7E
    deq = dequant_block(codes, scales, 128, 128)
    bound = np.abs(x) * 2.0 ** -4 + np.repeat(np.repeat(scales, 128, 0), 128, 1) * 2.0 ** -10
    assert np.all(np.abs(deq - x) <= bound * (1 + 1e-12))


def test_mx_quant_properties():
    x = synthetic.normal(0, synthetic.TID_A, 0, (64, 256))
    x[3, 32:64] = 0.0                              # an all-zero group
    x[5, 0:32] = np.float32(0.5)
    x[5, 7] = np.float32(448.0 * 2.0 ** -3)       # amax exactly a power of two of 448
    codes, e8 = oracle.quant_mx(x)
    assert e8.shape == (64, 8)
    assert e8[3, 1] == 0 and np.all(codes[3, 32:64] == 0)
    assert e8[5, 0] == 127 - 3 and codes[5, 7] == 0x7E
    assert TABLE[codes[5, 0]] * 2.0 ** -3 == 0.5
    scale = np.exp2(np.repeat(e8.astype(np.float64) - 127, 32, axis=1))
    deq = TABLE[codes] * scale
    nz = np.repeat(e8 > 0, 32, axis=1)
    bound = np.abs(x) * 2.0 ** -4 + scale * 2.0 ** -10
    assert np.all(np.abs(deq - x)[nz] <= bound[nz] * (1 + 1e-12))
    # power-of-two scale never lets a code exceed the format: all |codes| <= 448
    assert np.all(np.abs(TABLE[codes]) <= 448)


def test_bf16_rows_at_exact_midpoints_match_library_cast(payload):
    """bf16-valued rows put many x * 448 / amax exactly on an e4m3 rounding midpoint
    (both are numbers with few significant bits).  There the code depends on
    both fp32 roundings of the encoding, s = fp32(amax / 448) and fp32(x / s)
    (the scale rule of MORI GEMM + All-Reduce Benchmark, 'The fp8 wire'), so
    the oracle's quantisers are held to PyTorch's fp32 division and float8
    cast on such rows, which hold over 1% exact midpoints."""
    xb = torch.from_numpy(payload[:256]).to(torch.bfloat16).float()
    x = xb.numpy()
    g = xb.view(256, -1, 128)
    s_ref = g.abs().amax(dim=2) / torch.tensor(448.0, dtype=torch.float32)
    q_ref = (g / s_ref[:, :, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).reshape(256, -1)
    q, s = oracle.quant_block(x, 1, 128)
    assert np.array_equal(s, s_ref.numpy()) and np.array_equal(q, q_ref.numpy())
    # how many values sit exactly on a midpoint next to their code (products of few-bit numbers are exact)
    xa = np.abs(x.reshape(256, -1, 128).astype(np.float64))
    am = xa.max(axis=2, keepdims=True)
    c = q.reshape(xa.shape).astype(np.int64) & 0x7F
    v = np.abs(TABLE[c])
    lo, hi = np.abs(TABLE[np.clip(c - 1, 0, 126)]), np.abs(TABLE[np.clip(c + 1, 0, 126)])
    mid = (xa > 0) & ((xa * 448.0 == (v + lo) / 2 * am) | (xa * 448.0 == (v + hi) / 2 * am))
    assert mid.mean() > 0.01
    qr, sr = oracle.rowquant(x)
    sr_ref = xb.abs().amax(dim=1) / torch.tensor(448.0, dtype=torch.float32)
    qr_ref = (xb / sr_ref[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(sr, sr_ref.numpy()) and np.array_equal(qr, qr_ref)


def test_two_roundings_at_a_midpoint_closed_form():
    """Worked by hand in exact arithmetic.  amax = 3.5 gives s = 2^-7 exactly:
    3.375 / s = 432 ties between 416 (0x7D) and 448 (0x7E) and takes the even
    code 0x7E; 3.125 / s = 400 ties between 384 (0x7C) and 416 and takes 0x7C.
    amax = 2.03125 = 2 + 2^-5 gives s = fp32(amax / 448) just below amax / 448,
    so x = 0.0029754638671875 (a bf16 value, x * 448 / amax = 0.65625 exactly)
    has x / s a little above the midpoint 0.65625 of 0.625 (0x32) and 0.6875
    (0x33), by less than half an fp32 step: fp32(x / s) is the midpoint itself
    and ties to the even code 0x32.  Rounding the exact quotient straight to
    e4m3 would give 0x33."""
    x = np.array([[3.5, 3.375, 3.125, -3.375], [2.03125, 0.0029754638671875, -0.0029754638671875, 1.0]],
                 dtype=np.float32)
    q, s = oracle.rowquant(x)
    assert s[0] == np.float32(2.0 ** -7)
    assert list(q[0]) == [0x7E, 0x7E, 0x7C, 0xFE]
    assert np.float32(2.03125) / np.float32(448.0) == s[1] and np.float64(s[1]) < 2.03125 / 448.0
    assert q[1, 1] == 0x32 and q[1, 2] == 0xB2
    qb, sb = oracle.quant_block(x, 1, 4)
    assert np.array_equal(qb, q) and np.array_equal(sb[:, 0], s)
