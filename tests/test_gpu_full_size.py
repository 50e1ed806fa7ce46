"""Parity at the full workload sizes, in the launch configuration the
benchmark times (fused_gemm_reduce, bands = P), on sampled output rows the
oracle computes one by one: the first, second, middle and last rows of every
band plus random rows, all columns.

  - wo_b prefill: P=8, A_p [4096, 2048], B_p [7168, 2048], blockscale
  - wo_b full chunk: the same at M = 8192 and M = 16384 (the headline shape)
  - fp8 wire on the M = 16384 output
  - mxfp8: P=4, A_p [16384, 2048], B_p [7168, 2048], ue8m0 1x32
  - the band path's in-kernel reduce against GEMMAR_SERIAL_REDUCE, bitwise

Operands are drawn by `synthetic` and quantised by the oracle on the host, so
both sides consume identical codes and scales.  The M=4096 and M=8192 cases
use the leading rows of the M=16384 operands (same generator streams).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import PAGES_BF16_WIRE_REL_L2, blockscale_operands, check_bf16_output, mx_operands, rel_l2

pytestmark = pytest.mark.gpu

P, MMAX, N, K = 8, 16384, 7168, 2048


def sample_rows(M, bands, per_band_random=2, seed=0):
    rng = np.random.default_rng(seed)
    rpb = M // bands
    rows = []
    for b in range(bands):
        base = b * rpb
        rows += [base, base + 1, base + rpb // 2, base + rpb - 1]
        rows += list(base + rng.integers(0, rpb, per_band_random))
    return np.unique(np.array(rows, dtype=np.int64))


@pytest.fixture(scope="module")
def g():
    import block_scaled_fp8_gemm_gb300 as g
    return g


@pytest.fixture(scope="module")
def headline(g):
    A, sa, B, sb = blockscale_operands(P, MMAX, N, K, seed=0)
    torch.cuda.set_device(0)
    dev = lambda a: torch.from_numpy(a).cuda()
    d = dict(A=A, sa=sa, B=B, sb=sb, dA=[dev(a) for a in A], dsa=[dev(s) for s in sa],
             dB=[dev(b) for b in B], dsb=[dev(s) for s in sb])
    ctx = g.gemmar_create(0, MMAX, N, K, P)
    d["ctx"] = ctx
    yield d
    ctx.close()


def run_fused(g, d, M, flags=0):
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.fused_gemm_reduce(d["ctx"], [a[:M] for a in d["dA"]], [s[:M] for s in d["dsa"]], d["dB"], d["dsb"],
                        out, bands=P, flags=flags)
    torch.cuda.synchronize()
    code, detail = g.gemmar_status(d["ctx"])
    assert code == 0, (code, detail)
    return out


def oracle_rows(d, M, rows):
    return oracle.gemm_reduce([a[:M] for a in d["A"]], [s[:M] for s in d["sa"]], d["B"], d["sb"], 0, rows=rows)


@pytest.mark.parametrize("M", [4096, 8192, 16384])
def test_fused_blockscale_full_size(g, headline, M):
    rows = sample_rows(M, P, seed=M)
    out = run_fused(g, headline, M)
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    ref, _ = oracle_rows(headline, M, rows)
    rl = check_bf16_output(got, ref, f"fused P=8 M={M} N={N} K={K}")
    assert rl < PAGES_BF16_WIRE_REL_L2      # below the pages' bf16-partial level, as fp32 partials should be
    # every output written, nothing non-finite anywhere
    assert torch.isfinite(out.float()).all()


def test_fused_slice_loop_full_size(g, headline):
    M = MMAX
    rows = sample_rows(M, P, seed=7)
    out = run_fused(g, headline, M, flags=g.GEMMAR_FUSE_SLICES)
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    ref, _ = oracle_rows(headline, M, rows)
    check_bf16_output(got, ref, f"fused slice loop P=8 M={M}")
    assert torch.isfinite(out.float()).all()


def test_fused_full_size_is_deterministic(g, headline):
    a = run_fused(g, headline, MMAX)
    b = run_fused(g, headline, MMAX, flags=g.GEMMAR_DEBUG_CANARY)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_fp8_wire_full_size(g, headline):
    M = MMAX
    rows = sample_rows(M, P, seed=3)
    wire = run_fused(g, headline, M, flags=g.GEMMAR_FP8_WIRE)
    got = wire[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    ref, ref16 = oracle_rows(headline, M, rows)
    q, s = oracle.rowquant(oracle.bf16_to_f32(ref16))
    wire_ref = oracle.bf16_to_f32(oracle.rowdequant(q, s))
    assert rel_l2(got, ref) <= 3e-2
    assert rel_l2(got, wire_ref) <= 1e-2
    # the band reduce quantising the rows itself gives the same bits
    fused = run_fused(g, headline, M, flags=g.GEMMAR_FP8_WIRE | g.GEMMAR_FUSE_QUANTIZE)
    assert torch.equal(fused.view(torch.int16), wire.view(torch.int16))


def test_fused_mx_full_size(g):
    Pm, M = 4, MMAX
    A, ea, B, eb = mx_operands(Pm, M, N, K, seed=4)
    torch.cuda.set_device(0)
    dev = lambda a: torch.from_numpy(a).cuda()
    ctx = g.gemmar_create(0, M, N, K, Pm)
    try:
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        g.fused_gemm_reduce(ctx, [dev(a) for a in A], [dev(s) for s in ea], [dev(b) for b in B],
                            [dev(s) for s in eb], out, scale_kind=g.GEMMAR_SCALE_MX32, bands=Pm)
        torch.cuda.synchronize()
        assert g.gemmar_status(ctx)[0] == 0
        ov, tot = g.gemmar_overlap_stats(ctx)   # part of it summed while the GEMM ran
        assert 0 < ov < tot, (ov, tot)
        rows = sample_rows(M, Pm, seed=5)
        got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy()
        ref, _ = oracle.gemm_reduce(A, ea, B, eb, 1, rows=rows)
        check_bf16_output(got, ref, f"fused mx P=4 M={M} N={N} K={K}")
        assert torch.isfinite(out.float()).all()
        # the slices summed on chip reproduce the band path's bits
        onchip = torch.empty_like(out)
        g.fused_gemm_reduce(ctx, [dev(a) for a in A], [dev(s) for s in ea], [dev(b) for b in B],
                            [dev(s) for s in eb], onchip, scale_kind=g.GEMMAR_SCALE_MX32, bands=Pm,
                            flags=g.GEMMAR_FUSE_ONCHIP)
        torch.cuda.synchronize()
        assert g.gemmar_status(ctx)[0] == 0
        assert torch.equal(onchip.view(torch.int16), out.view(torch.int16))
    finally:
        ctx.close()


@pytest.mark.parametrize("M", [4096, 16384])
def test_band_path_overlap_full_size(g, headline, M):
    """At the benchmark's shapes the GEMM kernel's reducer warps take a share of
    the bands while the GEMM runs; the output is bit-equal to leaving every
    block to band_reduce (GEMMAR_SERIAL_REDUCE)."""
    over = run_fused(g, headline, M)
    ov, tot = g.gemmar_overlap_stats(headline["ctx"])
    assert tot == P * (M // P // 128) * (N // 256) * 4 * 8
    assert 0 < ov < tot, (ov, tot)
    serial = run_fused(g, headline, M, flags=g.GEMMAR_SERIAL_REDUCE)
    assert torch.equal(over.view(torch.int16), serial.view(torch.int16))
    # an output base that is 16- but not 32-byte aligned takes the reducers' 16-byte stores
    base = torch.empty(M * N + 8, dtype=torch.bfloat16, device="cuda")
    shifted = base[8:].view(M, N)
    assert shifted.data_ptr() % 32 == 16
    g.fused_gemm_reduce(headline["ctx"], [a[:M] for a in headline["dA"]], [s[:M] for s in headline["dsa"]],
                        headline["dB"], headline["dsb"], shifted, bands=P)
    torch.cuda.synchronize()
    assert g.gemmar_status(headline["ctx"])[0] == 0
    assert g.gemmar_overlap_stats(headline["ctx"])[0] > 0
    assert torch.equal(shifted.view(torch.int16), over.view(torch.int16))


def test_onchip_full_size_bit_equal_to_pair_band_path(g, headline):
    """GEMMAR_FUSE_ONCHIP at the headline shape: sampled rows against the oracle,
    and the whole output bit-equal to the band path of the CTA-pair kernel and to
    the default one-CTA band path (the benchmark's headline step)."""
    M = MMAX
    band_one_cta = run_fused(g, headline, M)
    ctx2 = g.gemmar_create(0, M, N, K, P, flags=g.GEMMAR_CTA_PAIR)
    try:
        outs = []
        for flags in (g.GEMMAR_FUSE_ONCHIP, 0):
            out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            g.fused_gemm_reduce(ctx2, headline["dA"], headline["dsa"], headline["dB"], headline["dsb"], out,
                                bands=P, flags=flags)
            torch.cuda.synchronize()
            assert g.gemmar_status(ctx2)[0] == 0
            outs.append(out)
        assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
        assert torch.equal(outs[0].view(torch.int16), band_one_cta.view(torch.int16))
        rows = sample_rows(M, P, seed=11)
        got = outs[0][torch.from_numpy(rows).cuda()].float().cpu().numpy()
        ref, _ = oracle_rows(headline, M, rows)
        check_bf16_output(got, ref, f"on-chip P=8 M={M}")
    finally:
        ctx2.close()


def test_fused_ptpc_full_size(g):
    """ptpc at the headline shape: sampled rows against the oracle, the on-chip
    sums bit-equal to the band path."""
    from helpers import ptpc_operands
    A, sa, B, sb = ptpc_operands(P, MMAX, N, K, seed=12)
    torch.cuda.set_device(0)
    dev = lambda a: torch.from_numpy(a).cuda()
    ctx = g.gemmar_create(0, MMAX, N, K, P)
    try:
        outs = []
        for flags in (0, g.GEMMAR_FUSE_ONCHIP):
            out = torch.empty((MMAX, N), dtype=torch.bfloat16, device="cuda")
            g.fused_gemm_reduce(ctx, [dev(a) for a in A], [dev(s) for s in sa], [dev(b) for b in B],
                                [dev(s) for s in sb], out, scale_kind=g.GEMMAR_SCALE_PTPC, bands=P, flags=flags)
            torch.cuda.synchronize()
            assert g.gemmar_status(ctx)[0] == 0
            if flags == 0:
                ov, tot = g.gemmar_overlap_stats(ctx)   # part of it summed while the GEMM ran
                assert 0 < ov < tot, (ov, tot)
            outs.append(out)
        assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
        rows = sample_rows(MMAX, P, seed=13)
        got = outs[0][torch.from_numpy(rows).cuda()].float().cpu().numpy()
        ref, _ = oracle.gemm_reduce(A, sa, B, sb, 2, rows=rows)
        check_bf16_output(got, ref, f"ptpc P=8 M={MMAX}")
    finally:
        ctx.close()
