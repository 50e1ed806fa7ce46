"""GPU parity of the tcgen05 GEMMs and the fused GEMM + band reduce against the
fp64 oracle, through the C ABI, at sizes that span several tiles and ragged
tails; plus the fused path's determinism and its bitwise equality with the
split path (GEMM per slice into fp32 partials, then band_reduce)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import (PAGES_BF16_WIRE_REL_L2, blockscale_operands, check_bf16_output,
                     check_f32_output, mx_operands, ptpc_operands, rel_l2)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import block_scaled_fp8_gemm_gb300 as g
    return g


@pytest.fixture(scope="module")
def ctx(g):
    torch.cuda.set_device(0)
    c = g.gemmar_create(0, 1024, 1024, 512, 8, flags=g.GEMMAR_NO_SELF_TEST, wait_timeout_ns=1_000_000_000)
    yield c
    c.close()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def status_ok(g, ctx):
    torch.cuda.synchronize()
    code, detail = g.gemmar_status(ctx)
    assert code == 0, f"device status {code} at site {detail}"


# ------------------------------------------------------------ single-slice GEMMs

@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 256), (200, 384, 512), (384, 768, 384),
                                   (64, 256, 256), (1, 128, 128)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_blockscale(g, ctx, M, N, K, out_dtype):
    A, sa, B, sb = blockscale_operands(1, M, N, K, seed=M + N + K)
    ref, ref16 = oracle.gemm_reduce(A, sa, B, sb, 0)
    C = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    g.gemm_blockscale_fp8(ctx, dev(A[0]), dev(sa[0]), dev(B[0]), dev(sb[0]), C)
    status_ok(g, ctx)
    if out_dtype == torch.float32:
        check_f32_output(C.cpu().numpy(), ref, f"blockscale f32 {M}x{N}x{K}")
    else:
        check_bf16_output(C.float().cpu().numpy(), ref, f"blockscale bf16 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 448, 256), (200, 384, 512), (128, 896, 128),
                                   (1, 128, 256)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_mxfp8(g, ctx, M, N, K, out_dtype):
    A, ea, B, eb = mx_operands(1, M, N, K, seed=M + N + K)
    ref, _ = oracle.gemm_reduce(A, ea, B, eb, 1)
    C = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    g.gemm_mxfp8(ctx, dev(A[0]), dev(ea[0]), dev(B[0]), dev(eb[0]), C)
    status_ok(g, ctx)
    if out_dtype == torch.float32:
        check_f32_output(C.cpu().numpy(), ref, f"mx f32 {M}x{N}x{K}")
    else:
        check_bf16_output(C.float().cpu().numpy(), ref, f"mx bf16 {M}x{N}x{K}")


def test_gemm_zero_scale_rows_and_blocks(g, ctx):
    M, N, K = 256, 512, 256
    A, sa, B, sb = blockscale_operands(1, M, N, K, seed=77)
    sa[0][5, :] = 0.0          # a zero row: exact zeros
    sb[0][2, :] = 0.0          # B block-row 2: columns 256..383 exactly zero
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g.gemm_blockscale_fp8(ctx, dev(A[0]), dev(sa[0]), dev(B[0]), dev(sb[0]), C)
    status_ok(g, ctx)
    c = C.cpu().numpy()
    assert np.all(c[5] == 0) and np.all(c[:, 256:384] == 0)
    check_f32_output(c, ref, "zero scales")


# ------------------------------------------------------------ fused GEMM + reduce

def run_fused(g, ctx, A, sa, B, sb, kind, bands, flags=0):
    M, N = A[0].shape[0], B[0].shape[0]
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.fused_gemm_reduce(ctx, [dev(a) for a in A], [dev(s) for s in sa], [dev(b) for b in B],
                        [dev(s) for s in sb], out, scale_kind=kind, bands=bands, flags=flags)
    status_ok(g, ctx)
    return out


@pytest.mark.parametrize("P,M,N,K,bands", [(2, 256, 512, 256, 2),      # the tiny configuration
                                           (4, 512, 768, 256, 4),
                                           (3, 600, 384, 384, 3),      # ragged bands (200 rows)
                                           (8, 1024, 256, 128, 8),
                                           (2, 256, 512, 256, 1),
                                           (1, 384, 512, 256, 3),      # one slice: the reduce is a rounding
                                           (5, 1000, 640, 256, 8)])    # ragged: 125-row bands, 5 slices
def test_fused_blockscale_vs_oracle(g, ctx, P, M, N, K, bands):
    A, sa, B, sb = blockscale_operands(P, M, N, K, seed=P * M)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
    out = run_fused(g, ctx, A, sa, B, sb, g.GEMMAR_SCALE_BLOCK128, bands, flags=g.GEMMAR_DEBUG_CANARY)
    rl = check_bf16_output(out.float().cpu().numpy(), ref, f"fused P={P} M={M} N={N} K={K} bands={bands}")
    assert rl < PAGES_BF16_WIRE_REL_L2      # fp32 partials stay below the pages' bf16-partial level


@pytest.mark.parametrize("P,M,N,K,bands", [(2, 256, 448, 256, 2), (4, 384, 256, 128, 4), (3, 600, 384, 256, 3)])
def test_fused_mx_vs_oracle(g, ctx, P, M, N, K, bands):
    A, ea, B, eb = mx_operands(P, M, N, K, seed=P * M + 1)
    ref, _ = oracle.gemm_reduce(A, ea, B, eb, 1)
    out = run_fused(g, ctx, A, ea, B, eb, g.GEMMAR_SCALE_MX32, bands, flags=g.GEMMAR_DEBUG_CANARY)
    check_bf16_output(out.float().cpu().numpy(), ref, f"fused mx P={P} M={M} N={N} K={K}")


@pytest.mark.parametrize("K", [640, 768, 1152])
def test_mx_scale_groups_with_a_partial_group(g, K):
    """The mx kernel loads and copies the scale images of four K-blocks (4 x 128
    of K) at a time; K/128 = 5, 6 or 9 leaves a last group of 1, 2 or 1 blocks.
    Single GEMM against the oracle, the band path against the oracle, and the
    on-chip sums bit-equal to the band path."""
    P, M, N, bands = 3, 384, 448, 3
    c = g.gemmar_create(0, M, N, K, P, flags=g.GEMMAR_NO_SELF_TEST, wait_timeout_ns=1_000_000_000)
    try:
        A, ea, B, eb = mx_operands(P, M, N, K, seed=K + 3)
        one, _ = oracle.gemm_reduce(A[:1], ea[:1], B[:1], eb[:1], 1)
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        g.gemm_mxfp8(c, dev(A[0]), dev(ea[0]), dev(B[0]), dev(eb[0]), C)
        status_ok(g, c)
        check_f32_output(C.cpu().numpy(), one, f"mx f32 {M}x{N}x{K}")
        ref, _ = oracle.gemm_reduce(A, ea, B, eb, 1)
        band = run_fused(g, c, A, ea, B, eb, g.GEMMAR_SCALE_MX32, bands, flags=g.GEMMAR_DEBUG_CANARY)
        check_bf16_output(band.float().cpu().numpy(), ref, f"fused mx P={P} M={M} N={N} K={K}")
        onchip = run_fused(g, c, A, ea, B, eb, g.GEMMAR_SCALE_MX32, bands, flags=g.GEMMAR_FUSE_ONCHIP)
        assert torch.equal(onchip.view(torch.int16), band.view(torch.int16))
        slices = run_fused(g, c, A, ea, B, eb, g.GEMMAR_SCALE_MX32, bands, flags=g.GEMMAR_FUSE_SLICES)
        check_bf16_output(slices.float().cpu().numpy(), ref, f"mx slice loop K={K}")
    finally:
        c.close()


@pytest.mark.parametrize("kind", [0, 1])
def test_fused_equals_split_bitwise_and_is_deterministic(g, ctx, kind):
    P, M, N, K, bands = 4, 512, 512, 256, 4
    ops = blockscale_operands(P, M, N, K, seed=5) if kind == 0 else mx_operands(P, M, N, K, seed=5)
    A, sa, B, sb = ops
    out1 = run_fused(g, ctx, A, sa, B, sb, kind, bands)
    out2 = run_fused(g, ctx, A, sa, B, sb, kind, bands)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16)), "fused run is not deterministic"
    # split path: each slice's fp32 GEMM, arranged as W[band][p], then band_reduce
    rpb = M // bands
    W = torch.empty((bands, P, rpb, N), dtype=torch.float32, device="cuda")
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    gemm = g.gemm_blockscale_fp8 if kind == 0 else g.gemm_mxfp8
    for p in range(P):
        gemm(ctx, dev(A[p]), dev(sa[p]), dev(B[p]), dev(sb[p]), C)
        W[:, p] = C.view(bands, rpb, N)
    split = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.band_reduce(ctx, W, P, M, N, bands, split)
    status_ok(g, ctx)
    assert torch.equal(out1.view(torch.int16), split.view(torch.int16)), "fused != split"


@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("P,M,N,K,bands", [(8, 1024, 1024, 512, 8), (3, 600, 896, 384, 3)])
def test_band_path_overlap_equals_serial_reduce(g, ctx, kind, P, M, N, K, bands):
    """The band path's in-kernel reduce (spare GEMM warps summing complete bands
    while the GEMM runs) against the same call with every block left to
    band_reduce: bit-equal, within the tolerance of the oracle, and the block
    accounting consistent (blockscale, mx and ptpc kernels)."""
    make = (blockscale_operands, mx_operands, ptpc_operands)[kind]
    A, sa, B, sb = make(P, M, N, K, seed=P + M)
    over = run_fused(g, ctx, A, sa, B, sb, kind, bands, flags=g.GEMMAR_DEBUG_CANARY)
    ov, tot = g.gemmar_overlap_stats(ctx)
    wide = 224 if kind == 1 else 256
    bn = wide if N % wide == 0 else 128
    assert tot == bands * ((M // bands + 127) // 128) * (N // bn) * 4 * (bn // 32)
    assert 0 <= ov <= tot
    serial = run_fused(g, ctx, A, sa, B, sb, kind, bands, flags=g.GEMMAR_SERIAL_REDUCE | g.GEMMAR_DEBUG_CANARY)
    assert g.gemmar_overlap_stats(ctx) == (0, 0)
    run_fused(g, ctx, A, sa, B, sb, kind, bands, flags=g.GEMMAR_FUSE_SLICES)   # no band path: nothing to report
    assert g.gemmar_overlap_stats(ctx) == (0, 0)
    assert torch.equal(over.view(torch.int16), serial.view(torch.int16))
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, kind)
    check_bf16_output(over.float().cpu().numpy(), ref, f"overlapped band path kind={kind} P={P} M={M}")


@pytest.fixture(scope="module")
def ctx_wide(g):
    torch.cuda.set_device(0)
    c = g.gemmar_create(0, 1024, 2048, 384, 8, flags=g.GEMMAR_NO_SELF_TEST, wait_timeout_ns=1_000_000_000)
    yield c
    c.close()


@pytest.mark.parametrize("N,K", [(2048, 128), (2048, 256), (2048, 384), (1920, 128), (1920, 256)])
def test_band_path_short_k_several_tiles_per_cta(g, ctx_wide, N, K):
    """One, two and three K-blocks per tile with three or more tiles per CTA (512
    tiles of 256 columns, or 960 of 128 columns when N is not a multiple of 256,
    on at most 152 CTAs).  The one-CTA kernel parks each tile's sums in the TMEM
    buffer of its last K-block for the store warps; with fewer K-blocks than its
    usual single-buffered lead the hand-over takes its capped form.  Against the
    oracle, bit-equal to the same call with the reduce after the GEMM, and twice
    the same bits."""
    P, M, bands = 8, 1024, 4
    A, sa, B, sb = blockscale_operands(P, M, N, K, seed=K + N + 17)
    kind = g.GEMMAR_SCALE_BLOCK128
    band = run_fused(g, ctx_wide, A, sa, B, sb, kind, bands, flags=g.GEMMAR_DEBUG_CANARY)
    ov, tot = g.gemmar_overlap_stats(ctx_wide)
    bn = 256 if N % 256 == 0 else 128
    assert tot == bands * 2 * (N // bn) * 4 * (bn // 32) and 0 <= ov <= tot
    again = run_fused(g, ctx_wide, A, sa, B, sb, kind, bands)
    serial = run_fused(g, ctx_wide, A, sa, B, sb, kind, bands,
                       flags=g.GEMMAR_SERIAL_REDUCE | g.GEMMAR_DEBUG_CANARY)
    assert torch.equal(band.view(torch.int16), again.view(torch.int16))
    assert torch.equal(band.view(torch.int16), serial.view(torch.int16))
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
    check_bf16_output(band.float().cpu().numpy(), ref, f"band path N={N} K={K} (3 or more tiles per CTA)")


def test_fused_fp8_wire(g, ctx):
    P, M, N, K = 2, 256, 512, 256
    A, sa, B, sb = blockscale_operands(P, M, N, K, seed=9)
    ref, ref16 = oracle.gemm_reduce(A, sa, B, sb, 0)
    plain = run_fused(g, ctx, A, sa, B, sb, 0, P)
    wire = run_fused(g, ctx, A, sa, B, sb, 0, P, flags=g.GEMMAR_FP8_WIRE)
    # against the oracle's own chain: fp64 sum -> bf16 -> per-row e4m3 codec
    q_ref, s_ref = oracle.rowquant(oracle.bf16_to_f32(ref16))
    wire_ref = oracle.bf16_to_f32(oracle.rowdequant(q_ref, s_ref))
    w = wire.float().cpu().numpy()
    assert rel_l2(w, ref) <= 3e-2
    assert rel_l2(w, wire_ref) <= 1e-2
    # the wire is exactly the GPU codec applied to the GPU's reduced rows
    q = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    s = torch.empty((M,), dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.rowquant_e4m3(ctx, plain, q, s)
    g.rowdequant_e4m3(ctx, q, s, y)
    status_ok(g, ctx)
    assert torch.equal(y.view(torch.int16), wire.view(torch.int16))


@pytest.mark.parametrize("N", [12288, 12544])
def test_fused_quantize_at_its_width_limit(g, N):
    """The folded quantiser parks 8 bf16 rows of N in shared memory, N <= 12288
    (192 KB at the limit); above it the flag is ignored.  Either way the output
    is the unfolded wire's, bit for bit."""
    P, M, K, bands = 2, 256, 256, 2
    c = g.gemmar_create(0, M, N, K, P, flags=g.GEMMAR_NO_SELF_TEST, wait_timeout_ns=1_000_000_000)
    try:
        A, sa, B, sb = blockscale_operands(P, M, N, K, seed=N)
        kind = g.GEMMAR_SCALE_BLOCK128
        wire = run_fused(g, c, A, sa, B, sb, kind, bands, flags=g.GEMMAR_FP8_WIRE)
        fold = run_fused(g, c, A, sa, B, sb, kind, bands, flags=g.GEMMAR_FP8_WIRE | g.GEMMAR_FUSE_QUANTIZE)
        assert torch.equal(wire.view(torch.int16), fold.view(torch.int16))
    finally:
        c.close()


@pytest.mark.parametrize("serial", [False, True])
@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("P,M,N,K,bands", [(8, 1024, 1024, 512, 8), (3, 600, 896, 384, 3), (2, 256, 512, 256, 2)])
def test_fused_quantize_wire_equals_unfused_wire(g, ctx, kind, P, M, N, K, bands, serial):
    """GEMMAR_FUSE_QUANTIZE (the band reduce codes each group of 8 summed rows
    itself, taking the bf16 sums of blocks the GEMM kernel already reduced from
    the output) against the unfolded fp8 wire: bit-equal, with and without the
    in-kernel reduce, ragged bands included; and within the wire tolerance of
    the oracle."""
    make = (blockscale_operands, mx_operands, ptpc_operands)[kind]
    A, sa, B, sb = make(P, M, N, K, seed=3 * P + M)
    base = g.GEMMAR_FP8_WIRE | g.GEMMAR_DEBUG_CANARY | (g.GEMMAR_SERIAL_REDUCE if serial else 0)
    plain = run_fused(g, ctx, A, sa, B, sb, kind, bands, flags=base)
    fused = run_fused(g, ctx, A, sa, B, sb, kind, bands, flags=base | g.GEMMAR_FUSE_QUANTIZE)
    assert torch.equal(fused.view(torch.int16), plain.view(torch.int16))
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, kind)
    assert rel_l2(fused.float().cpu().numpy(), ref) <= 3e-2


@pytest.mark.parametrize("kind,P,M,N,K", [(0, 2, 256, 512, 256), (0, 3, 600, 384, 384), (0, 8, 512, 256, 128),
                                          (1, 2, 256, 448, 256), (1, 3, 300, 256, 256)])
def test_fused_slice_loop_vs_oracle_and_deterministic(g, ctx, kind, P, M, N, K):
    ops = blockscale_operands(P, M, N, K, seed=11 + P) if kind == 0 else mx_operands(P, M, N, K, seed=11 + P)
    A, sa, B, sb = ops
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, kind)
    out1 = run_fused(g, ctx, A, sa, B, sb, kind, P, flags=g.GEMMAR_FUSE_SLICES | g.GEMMAR_DEBUG_CANARY)
    out2 = run_fused(g, ctx, A, sa, B, sb, kind, P, flags=g.GEMMAR_FUSE_SLICES)
    check_bf16_output(out1.float().cpu().numpy(), ref, f"slice loop kind={kind} P={P} M={M} N={N} K={K}")
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


# ------------------------------------------------------------ CTA-pair vs one-CTA kernel

@pytest.fixture(scope="module")
def ctx_pair(g):
    torch.cuda.set_device(0)
    c = g.gemmar_create(0, 1024, 1024, 512, 8, flags=g.GEMMAR_NO_SELF_TEST | g.GEMMAR_CTA_PAIR,
                        wait_timeout_ns=1_000_000_000)
    yield c
    c.close()


@pytest.mark.parametrize("P,M,N,K,bands", [(2, 256, 512, 256, 2), (3, 600, 384, 384, 3), (8, 1024, 256, 128, 8),
                                           (4, 520, 640, 256, 4)])
def test_pair_and_single_cta_kernels_agree(g, ctx, ctx_pair, P, M, N, K, bands):
    A, sa, B, sb = blockscale_operands(P, M, N, K, seed=P * M + 3)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
    pair = run_fused(g, ctx_pair, A, sa, B, sb, 0, bands, flags=g.GEMMAR_DEBUG_CANARY)
    one = run_fused(g, ctx, A, sa, B, sb, 0, bands, flags=g.GEMMAR_DEBUG_CANARY)
    check_bf16_output(pair.float().cpu().numpy(), ref, f"pair kernel P={P} M={M} N={N} K={K}")
    check_bf16_output(one.float().cpu().numpy(), ref, f"one-CTA kernel P={P} M={M} N={N} K={K}")
    # the same fp32 promotion order on both, and the tensor cores accumulate a
    # K-block the same way for M=256 pairs as for M=128: the same bits
    assert torch.equal(pair.view(torch.int16), one.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(200, 384, 512), (1, 128, 128), (384, 768, 384)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_pair_gemm_blockscale(g, ctx_pair, M, N, K, out_dtype):
    A, sa, B, sb = blockscale_operands(1, M, N, K, seed=M + 2 * N)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
    out = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    g.gemm_blockscale_fp8(ctx_pair, dev(A[0]), dev(sa[0]), dev(B[0]), dev(sb[0]), out)
    status_ok(g, ctx_pair)
    if out_dtype == torch.float32:
        check_f32_output(out.cpu().numpy(), ref, f"pair blockscale f32 M={M} N={N} K={K}")
    else:
        check_bf16_output(out.float().cpu().numpy(), ref, f"pair blockscale bf16 M={M} N={N} K={K}")


@pytest.mark.parametrize("P,M,N,K", [(2, 256, 512, 256), (3, 600, 384, 384)])
def test_pair_slice_loop(g, ctx_pair, P, M, N, K):
    A, sa, B, sb = blockscale_operands(P, M, N, K, seed=31 + P)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
    out = run_fused(g, ctx_pair, A, sa, B, sb, 0, P, flags=g.GEMMAR_FUSE_SLICES | g.GEMMAR_DEBUG_CANARY)
    check_bf16_output(out.float().cpu().numpy(), ref, f"pair slice loop P={P} M={M} N={N} K={K}")


# ------------------------------------------------------------ partials summed on chip

@pytest.mark.parametrize("P,M,N,K,bands", [(2, 256, 512, 256, 2), (3, 600, 768, 384, 3), (8, 1024, 256, 128, 8),
                                           (1, 384, 512, 256, 1), (4, 520, 1024, 256, 4), (4, 512, 512, 256, 1)])
def test_onchip_equals_band_path_bitwise(g, ctx_pair, P, M, N, K, bands):
    A, sa, B, sb = blockscale_operands(P, M, N, K, seed=41 + P * M)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
    onchip = run_fused(g, ctx_pair, A, sa, B, sb, 0, bands, flags=g.GEMMAR_FUSE_ONCHIP | g.GEMMAR_DEBUG_CANARY)
    band = run_fused(g, ctx_pair, A, sa, B, sb, 0, bands, flags=g.GEMMAR_DEBUG_CANARY)
    check_bf16_output(onchip.float().cpu().numpy(), ref, f"on-chip P={P} M={M} N={N} K={K}")
    # same per-slice fp32 partials, same summation order, one bf16 rounding
    assert torch.equal(onchip.view(torch.int16), band.view(torch.int16))
    again = run_fused(g, ctx_pair, A, sa, B, sb, 0, bands, flags=g.GEMMAR_FUSE_ONCHIP)
    assert torch.equal(onchip.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("kind,P,M,N,K", [(0, 2, 256, 384, 256), (1, 2, 256, 448, 256), (1, 3, 600, 384, 256),
                                          (1, 4, 384, 256, 128), (1, 1, 256, 448, 256), (1, 8, 512, 448, 128)])
def test_onchip_equals_band_path_default_context(g, ctx, kind, P, M, N, K):
    # blockscale with N % 256 != 0 takes the band path; mx sums its slices on chip
    # (a TMEM buffer per slice, the running sum in registers): bit-equal either way
    ops = blockscale_operands(P, M, N, K, seed=43 + P) if kind == 0 else mx_operands(P, M, N, K, seed=43 + P)
    A, sa, B, sb = ops
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, kind)
    a = run_fused(g, ctx, A, sa, B, sb, kind, P, flags=g.GEMMAR_FUSE_ONCHIP | g.GEMMAR_DEBUG_CANARY)
    b = run_fused(g, ctx, A, sa, B, sb, kind, P)
    check_bf16_output(a.float().cpu().numpy(), ref, f"on-chip kind={kind} P={P} M={M} N={N} K={K}")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_onchip_on_default_context_matches_one_cta_band_path(g, ctx):
    P, M, N, K = 4, 512, 768, 256
    A, sa, B, sb = blockscale_operands(P, M, N, K, seed=47)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
    onchip = run_fused(g, ctx, A, sa, B, sb, 0, P, flags=g.GEMMAR_FUSE_ONCHIP)
    band = run_fused(g, ctx, A, sa, B, sb, 0, P)
    check_bf16_output(onchip.float().cpu().numpy(), ref, "on-chip, default context")
    # the on-chip sums (CTA-pair kernel) reproduce the one-CTA band path's bits
    assert torch.equal(onchip.view(torch.int16), band.view(torch.int16))


# ------------------------------------------------------------ ptpc (per-token / per-channel scales)

@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (200, 384, 512), (384, 768, 384), (1, 128, 256),
                                   (256, 512, 1024)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_ptpc(g, ctx, M, N, K, out_dtype):
    from helpers import ptpc_operands
    A, sa, B, sb = ptpc_operands(1, M, N, K, seed=M + 3 * N + K)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 2)
    C = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    g.gemm_ptpc_fp8(ctx, dev(A[0]), dev(sa[0]), dev(B[0]), dev(sb[0]), C)
    status_ok(g, ctx)
    if out_dtype == torch.float32:
        check_f32_output(C.cpu().numpy(), ref, f"ptpc f32 {M}x{N}x{K}")
    else:
        check_bf16_output(C.float().cpu().numpy(), ref, f"ptpc bf16 {M}x{N}x{K}")


@pytest.mark.parametrize("P,M,N,K,bands", [(2, 256, 512, 256, 2), (3, 600, 384, 384, 3), (8, 1024, 256, 128, 8),
                                           (4, 520, 1024, 256, 4), (1, 256, 256, 256, 1)])
def test_fused_ptpc_band_onchip_bitwise(g, ctx, P, M, N, K, bands):
    from helpers import ptpc_operands
    A, sa, B, sb = ptpc_operands(P, M, N, K, seed=51 + P * M)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 2)
    band = run_fused(g, ctx, A, sa, B, sb, g.GEMMAR_SCALE_PTPC, bands, flags=g.GEMMAR_DEBUG_CANARY)
    rl = check_bf16_output(band.float().cpu().numpy(), ref, f"ptpc band P={P} M={M} N={N} K={K}")
    assert rl < PAGES_BF16_WIRE_REL_L2
    onchip = run_fused(g, ctx, A, sa, B, sb, g.GEMMAR_SCALE_PTPC, bands,
                       flags=g.GEMMAR_FUSE_ONCHIP | g.GEMMAR_DEBUG_CANARY)
    assert torch.equal(onchip.view(torch.int16), band.view(torch.int16))
    slices = run_fused(g, ctx, A, sa, B, sb, g.GEMMAR_SCALE_PTPC, bands, flags=g.GEMMAR_FUSE_SLICES)
    assert torch.equal(slices.view(torch.int16), band.view(torch.int16))


def test_ptpc_zero_scales_give_exact_zeros(g, ctx):
    from helpers import ptpc_operands
    P, M, N, K = 3, 384, 512, 256
    A, sa, B, sb = ptpc_operands(P, M, N, K, seed=61)
    for p in range(P):
        sa[p][17] = 0.0           # token 17 scaled to zero in every slice
        sb[p][300] = 0.0          # channel 300 scaled to zero in every slice
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, 2)
    for flags in (0, g.GEMMAR_FUSE_ONCHIP):
        out = run_fused(g, ctx, A, sa, B, sb, g.GEMMAR_SCALE_PTPC, P, flags=flags | g.GEMMAR_DEBUG_CANARY)
        o = out.float().cpu().numpy()
        assert np.all(o[17] == 0) and np.all(o[:, 300] == 0)
        check_bf16_output(o, ref, f"ptpc zero scales flags={flags}")


@pytest.mark.parametrize("kind", [0, 1, 2])
def test_fp8_wire_after_onchip_equals_wire_after_band_path(g, ctx, ctx_pair, kind):
    # the wire codec runs on the reduced rows, which the on-chip sums reproduce bit for bit
    from helpers import ptpc_operands
    P, M, N, K = 4, 512, 512, 256
    make = {0: blockscale_operands, 1: mx_operands, 2: ptpc_operands}[kind]
    A, sa, B, sb = make(P, M, N, K, seed=71 + kind)
    c = ctx_pair if kind == 0 else ctx
    band = run_fused(g, c, A, sa, B, sb, kind, P, flags=g.GEMMAR_FP8_WIRE)
    onchip = run_fused(g, c, A, sa, B, sb, kind, P, flags=g.GEMMAR_FP8_WIRE | g.GEMMAR_FUSE_ONCHIP)
    assert torch.equal(onchip.view(torch.int16), band.view(torch.int16))
    ref, ref16 = oracle.gemm_reduce(A, sa, B, sb, kind)
    assert rel_l2(onchip.float().cpu().numpy(), ref) <= 3e-2
