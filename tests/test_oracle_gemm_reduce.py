"""Pins for the oracle's scaled GEMM and P-way reduction (CPU only).

Checked against: the plain fp64 matrix product of the dequantised operands
(numpy, a textbook routine) for P = 1; exact rational brute force on small
inputs; power-of-two scale invariance; zero-scale blocks; the ordered fp32
reduction against numpy's fp32 arithmetic and PyTorch's bf16 cast.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synthetic
from test_oracle_e4m3 import bf16_nearest_bruteforce

TABLE = oracle.e4m3_decode_table()


def make_blockscale(P, M, N, K, seed=0):
    A, sa, B, sb = [], [], [], []
    for p in range(P):
        a, s = oracle.quant_act_1x128(synthetic.normal(seed, synthetic.TID_A, p, (M, K)))
        b, t = oracle.quant_weight_128x128(synthetic.normal(seed, synthetic.TID_B, p, (N, K), sigma=0.02))
        A.append(a); sa.append(s); B.append(b); sb.append(t)
    return A, sa, B, sb


def make_mx(P, M, N, K, seed=0):
    A, sa, B, sb = [], [], [], []
    for p in range(P):
        a, s = oracle.quant_mx(synthetic.normal(seed, synthetic.TID_A, p, (M, K)))
        b, t = oracle.quant_mx(synthetic.normal(seed, synthetic.TID_B, p, (N, K), sigma=0.02))
        A.append(a); sa.append(s); B.append(b); sb.append(t)
    return A, sa, B, sb


def dequant_bs(A, sa, B, sb):
    a = TABLE[A] * np.repeat(sa.astype(np.float64), 128, axis=1)
    b = TABLE[B] * np.repeat(np.repeat(sb.astype(np.float64), 128, axis=0), 128, axis=1)[:B.shape[0]]
    return a, b


def dequant_mx(A, ea, B, eb):
    a = TABLE[A] * np.exp2(np.repeat(ea.astype(np.float64) - 127, 32, axis=1))
    b = TABLE[B] * np.exp2(np.repeat(eb.astype(np.float64) - 127, 32, axis=1))
    return a, b


def test_p1_equals_plain_matmul_blockscale():
    A, sa, B, sb = make_blockscale(1, 96, 384, 512, seed=1)     # 3 B-scale blocks along N
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
    a, b = dequant_bs(A[0], sa[0], B[0], sb[0])
    plain = a @ b.T
    assert np.max(np.abs(ref - plain)) <= 1e-12 * np.max(np.abs(plain))


def test_p1_equals_plain_matmul_mx():
    A, sa, B, sb = make_mx(1, 64, 160, 256, seed=2)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 1)
    a, b = dequant_mx(A[0], sa[0], B[0], sb[0])
    plain = a @ b.T
    assert np.max(np.abs(ref - plain)) <= 1e-12 * np.max(np.abs(plain))


def test_p_way_sum_equals_sum_of_plain_matmuls():
    P = 3
    A, sa, B, sb = make_blockscale(P, 64, 256, 256, seed=3)
    ref, out = oracle.gemm_reduce(A, sa, B, sb, 0)
    plain = sum(np.matmul(*[dequant_bs(A[p], sa[p], B[p], sb[p])[0]],
                          dequant_bs(A[p], sa[p], B[p], sb[p])[1].T) for p in range(P))
    assert np.max(np.abs(ref - plain)) <= 1e-12 * np.max(np.abs(plain))
    # rows subset returns exactly the same rows
    rows = np.array([63, 0, 17])
    ref_s, out_s = oracle.gemm_reduce(A, sa, B, sb, 0, rows=rows)
    assert np.array_equal(ref_s, ref[rows]) and np.array_equal(out_s, out[rows])


def test_power_of_two_scale_invariance():
    A, sa, B, sb = make_blockscale(2, 32, 256, 256, seed=4)
    ref, out = oracle.gemm_reduce(A, sa, B, sb, 0)
    sa2 = [s * np.float32(8.0) for s in sa]
    sb2 = [s / np.float32(8.0) for s in sb]
    ref2, out2 = oracle.gemm_reduce(A, sa2, B, sb2, 0)
    assert np.array_equal(ref, ref2) and np.array_equal(out, out2)
    ref3, _ = oracle.gemm_reduce(A, [s * np.float32(2.0 ** -5) for s in sa], B, sb, 0)
    assert np.array_equal(ref3, ref * 2.0 ** -5)


def test_zero_scale_blocks_give_exact_zero_contribution():
    A, sa, B, sb = make_blockscale(1, 16, 256, 384, seed=5)
    sa0 = [sa[0].copy()]
    sa0[0][3, 1] = 0.0                    # row 3, K-block 1 scaled to zero
    A0 = [A[0].copy()]
    A0[0][3, 128:256] = 0                 # equivalent: zero codes in that block
    r1, _ = oracle.gemm_reduce(A, sa0, B, sb, 0)
    r2, _ = oracle.gemm_reduce(A0, sa, B, sb, 0)
    assert np.array_equal(r1, r2)
    sb0 = [sb[0].copy()]
    sb0[0][1, :] = 0.0                    # B block-row 1 (columns 128..255) scaled to zero
    r3, o3 = oracle.gemm_reduce(A, sa, B, sb0, 0)
    assert np.all(r3[:, 128:256] == 0) and np.all(o3[:, 128:256] == 0)
    sa_row = [sa[0].copy()]
    sa_row[0][7, :] = 0.0                 # an all-zero row
    r4, o4 = oracle.gemm_reduce(A, sa_row, B, sb, 0)
    assert np.all(r4[7] == 0) and np.all(o4[7] == 0)


def exact_blockscale(A, sa, B, sb):
    """Exact rational sum over slices, K-blocks and K of the scaled products."""
    P = len(A)
    M, K = A[0].shape
    N = B[0].shape[0]
    res = [[Fraction(0)] * N for _ in range(M)]
    mag = [[Fraction(0)] * N for _ in range(M)]      # sum of |terms|, for the rounding bound
    for p in range(P):
        for m in range(M):
            for n in range(N):
                for kb in range(K // 128):
                    dot = sum(Fraction(float(TABLE[A[p][m, k]])) * Fraction(float(TABLE[B[p][n, k]]))
                              for k in range(kb * 128, kb * 128 + 128))
                    term = Fraction(float(sa[p][m, kb])) * Fraction(float(sb[p][n // 128, kb])) * dot
                    res[m][n] += term
                    mag[m][n] += abs(term)
    return res, mag


def test_bruteforce_8x8x128_exact_rational():
    # 8x8 outputs, two slices of K = 128 and one slice-pair of K = 256 blocks
    for (P, K) in ((2, 128), (1, 256)):
        A, sa, B, sb = make_blockscale(P, 8, 8, K, seed=6 + K)
        ref, out = oracle.gemm_reduce(A, sa, B, sb, 0)
        exact, mag = exact_blockscale(A, sa, B, sb)
        for m in range(8):
            for n in range(8):
                assert out[m, n] == bf16_nearest_bruteforce(exact[m][n]), (m, n)
                # a few fp64 roundings (scale product, K-block and slice sums), each
                # bounded by 2^-53 of the magnitude it carries
                assert abs(Fraction(float(ref[m, n])) - exact[m][n]) <= mag[m][n] * Fraction(8, 2 ** 53)


def test_bruteforce_mx_exact_rational():
    A, sa, B, sb = make_mx(2, 4, 8, 64, seed=9)
    ref, out = oracle.gemm_reduce(A, sa, B, sb, 1)
    for m in range(4):
        for n in range(8):
            tot, mag = Fraction(0), Fraction(0)
            for p in range(2):
                for g in range(2):
                    dot = sum(Fraction(float(TABLE[A[p][m, k]])) * Fraction(float(TABLE[B[p][n, k]]))
                              for k in range(g * 32, g * 32 + 32))
                    term = dot * Fraction(2) ** (int(sa[p][m, g]) + int(sb[p][n, g]) - 254)
                    tot += term
                    mag += abs(term)
            assert out[m, n] == bf16_nearest_bruteforce(tot)
            assert abs(Fraction(float(ref[m, n])) - tot) <= mag * Fraction(8, 2 ** 53)


def test_slice_order_does_not_matter_in_fp64():
    A, sa, B, sb = make_blockscale(4, 32, 256, 256, seed=10)
    ref, out = oracle.gemm_reduce(A, sa, B, sb, 0)
    perm = [2, 0, 3, 1]
    ref2, out2 = oracle.gemm_reduce([A[i] for i in perm], [sa[i] for i in perm],
                                    [B[i] for i in perm], [sb[i] for i in perm], 0)
    assert np.max(np.abs(ref - ref2)) <= 1e-14 * np.max(np.abs(ref))
    assert np.mean(out != out2) < 1e-3


def test_reduce_f32_ordered_matches_numpy_and_library():
    rng = np.random.default_rng(11)
    W = (rng.standard_normal((8, 64, 256)) * np.exp2(rng.integers(-3, 3, (8, 64, 256)))).astype(np.float32)
    out = oracle.reduce_f32_ordered(W)
    s = W[0].copy()
    for p in range(1, 8):
        s = (s + W[p]).astype(np.float32)          # fp32 add, p ascending
    ref = torch.from_numpy(s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, ref)
    # P = 1 is the identity up to the bf16 rounding
    assert np.array_equal(oracle.reduce_f32_ordered(W[:1]),
                          torch.from_numpy(W[0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


# ------------------------------------------------------------------ ptpc (scale_kind 2)

def make_ptpc(P, M, N, K, seed=0):
    A, sa, B, sb = [], [], [], []
    for p in range(P):
        a, s = oracle.quant_ptpc(synthetic.normal(seed, synthetic.TID_A, p, (M, K)))
        b, t = oracle.quant_ptpc(synthetic.normal(seed, synthetic.TID_B, p, (N, K), sigma=0.02))
        A.append(a); sa.append(s); B.append(b); sb.append(t)
    return A, sa, B, sb


def test_ptpc_quantiser_is_the_row_codec():
    # per-token / per-channel scales are one group per row: the fp8-wire row codec
    x = synthetic.normal(3, synthetic.TID_X, 0, (40, 384))
    q1, s1 = oracle.quant_ptpc(x)
    q2, s2 = oracle.rowquant(x)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_p1_equals_plain_matmul_ptpc():
    A, sa, B, sb = make_ptpc(1, 72, 200, 384, seed=21)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 2)
    a = TABLE[A[0]] * sa[0].astype(np.float64)[:, None]
    b = TABLE[B[0]] * sb[0].astype(np.float64)[:, None]
    plain = a @ b.T
    assert np.max(np.abs(ref - plain)) <= 1e-12 * np.max(np.abs(plain))


def test_ptpc_with_unit_scales_equals_blockscale_with_unit_scales():
    # the two scale kinds agree where they describe the same operands
    A, _, B, _ = make_ptpc(2, 16, 256, 256, seed=22)
    one_a = [np.ones((16,), np.float32)] * 2
    one_b = [np.ones((256,), np.float32)] * 2
    r_pt, o_pt = oracle.gemm_reduce(A, one_a, B, one_b, 2)
    r_bs, o_bs = oracle.gemm_reduce(A, [np.ones((16, 2), np.float32)] * 2, B, [np.ones((2, 2), np.float32)] * 2, 0)
    assert np.max(np.abs(r_pt - r_bs)) <= 1e-13 * np.max(np.abs(r_bs))


def test_ptpc_scale_invariances_and_zero_rows():
    A, sa, B, sb = make_ptpc(2, 24, 256, 256, seed=23)
    ref, out = oracle.gemm_reduce(A, sa, B, sb, 2)
    ref2, out2 = oracle.gemm_reduce(A, [s * np.float32(4.0) for s in sa], B, [s / np.float32(4.0) for s in sb], 2)
    assert np.array_equal(ref, ref2) and np.array_equal(out, out2)
    sa0 = [s.copy() for s in sa]
    sb0 = [s.copy() for s in sb]
    for p in range(2):
        sa0[p][5] = 0.0                    # token 5 scaled to zero in every slice
        sb0[p][200] = 0.0                  # channel 200 scaled to zero in every slice
    r3, o3 = oracle.gemm_reduce(A, sa0, B, sb0, 2)
    assert np.all(r3[5] == 0) and np.all(o3[5] == 0)
    assert np.all(r3[:, 200] == 0) and np.all(o3[:, 200] == 0)


def test_bruteforce_ptpc_exact_rational():
    A, sa, B, sb = make_ptpc(2, 6, 8, 128, seed=24)
    ref, out = oracle.gemm_reduce(A, sa, B, sb, 2)
    for m in range(6):
        for n in range(8):
            tot, mag = Fraction(0), Fraction(0)
            for p in range(2):
                dot = sum(Fraction(float(TABLE[A[p][m, k]])) * Fraction(float(TABLE[B[p][n, k]])) for k in range(128))
                term = Fraction(float(sa[p][m])) * Fraction(float(sb[p][n])) * dot
                tot += term
                mag += abs(term)
            assert out[m, n] == bf16_nearest_bruteforce(tot)
            assert abs(Fraction(float(ref[m, n])) - tot) <= mag * Fraction(8, 2 ** 53)
