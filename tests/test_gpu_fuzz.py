"""Seeded random shapes inside the library's shape rules, for every scale kind.

For each shape the fused band path (with the in-kernel reduce of completed
bands) is checked against the fp64 oracle within the stated tolerance.  Every
other way of producing the same result is then checked against the band path
bit for bit:
  - the whole reduce after the GEMM (GEMMAR_SERIAL_REDUCE);
  - the on-chip sums (GEMMAR_FUSE_ONCHIP, which takes the band path itself
    for blockscale shapes the CTA-pair kernel does not cover);
  - blockscale on a GEMMAR_CTA_PAIR context (the CTA-pair kernel's band path
    where N % 256 == 0);
  - the fp8 wire, with and without the row quantiser folded into the reduce,
    both equal to the library's row codec applied to the band path's rows.
The draws include one-row bands, bands that end inside a tile, P = 1, and
N on both mxfp8 tile widths (multiples of 128 and of 224).

The single kernels get random shapes too: each scale kind's one-slice GEMM
with an fp32 output against the oracle, and the band reduce and the row codec
bit for bit against the oracle's fp32 ordered sum and row codec."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from helpers import blockscale_operands, check_bf16_output, check_f32_output, mx_operands, ptpc_operands

pytestmark = pytest.mark.gpu

MAX_M, MAX_N, MAX_K, MAX_P = 1024, 1024, 512, 8
CASES_PER_KIND = 24


def draw_shapes(kind, n, seed):
    """n shapes (P, M, N, K, bands) with M % bands == 0, N a multiple of 128
    (or of 224 for mxfp8), K a multiple of 128, sized so the oracle takes a
    second or two."""
    rng = np.random.RandomState(seed)
    n_choices = [c for c in range(128, MAX_N + 1, 32) if c % 128 == 0 or (kind == 1 and c % 224 == 0)]
    out = []
    while len(out) < n:
        P = int(rng.randint(1, MAX_P + 1))
        bands = int(rng.randint(1, 9))
        if rng.rand() < 0.4:
            rpb = int(rng.choice([1, 3, 64, 127, 128, 129, 200, 256]))
        else:
            rpb = int(rng.randint(1, MAX_M // bands + 1))
        M = bands * rpb
        N = int(rng.choice(n_choices))
        K = int(rng.choice([128, 256, 384, 512]))
        if M > MAX_M or P * M * N * K > 1_500_000_000:
            continue
        out.append((P, M, N, K, bands))
    return out


CASES = [(kind, *shape) for kind in (0, 1, 2) for shape in draw_shapes(kind, CASES_PER_KIND, 7100 + kind)]


@pytest.fixture(scope="module")
def g():
    import block_scaled_fp8_gemm_gb300 as g
    return g


@pytest.fixture(scope="module")
def ctx(g):
    torch.cuda.set_device(0)
    c = g.gemmar_create(0, MAX_M, MAX_N, MAX_K, MAX_P, flags=g.GEMMAR_NO_SELF_TEST,
                        wait_timeout_ns=1_000_000_000)
    yield c
    c.close()


@pytest.fixture(scope="module")
def ctx_pair(g):
    torch.cuda.set_device(0)
    c = g.gemmar_create(0, MAX_M, MAX_N, MAX_K, MAX_P, flags=g.GEMMAR_NO_SELF_TEST | g.GEMMAR_CTA_PAIR,
                        wait_timeout_ns=1_000_000_000)
    yield c
    c.close()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("kind,P,M,N,K,bands", CASES,
                         ids=[f"k{k}-P{P}-M{M}-N{N}-K{K}-b{b}" for k, P, M, N, K, b in CASES])
def test_random_shape(g, ctx, ctx_pair, kind, P, M, N, K, bands):
    make = (blockscale_operands, mx_operands, ptpc_operands)[kind]
    A, sa, B, sb = make(P, M, N, K, seed=P * 100003 + M * 31 + N + K)
    dA, dsa, dB, dsb = [dev(a) for a in A], [dev(s) for s in sa], [dev(b) for b in B], [dev(s) for s in sb]

    def fused(flags, c=ctx):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        g.fused_gemm_reduce(c, dA, dsa, dB, dsb, out, scale_kind=kind, bands=bands, flags=flags)
        torch.cuda.synchronize()
        code, detail = g.gemmar_status(c)
        assert code == 0, f"device status {code} at site {detail} (flags {flags:#x})"
        return out

    what = f"kind {kind} P={P} M={M} N={N} K={K} bands={bands}"
    band = fused(g.GEMMAR_DEBUG_CANARY)
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, kind)
    check_bf16_output(band.float().cpu().numpy(), ref, what)

    assert torch.equal(bits(fused(g.GEMMAR_SERIAL_REDUCE)), bits(band)), f"{what}: serial reduce != band path"
    assert torch.equal(bits(fused(g.GEMMAR_FUSE_ONCHIP)), bits(band)), f"{what}: on-chip != band path"
    if kind == 0:
        assert torch.equal(bits(fused(0, ctx_pair)), bits(band)), f"{what}: CTA-pair context != band path"

    q = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    s = torch.empty((M,), dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.rowquant_e4m3(ctx, band, q, s)
    g.rowdequant_e4m3(ctx, q, s, y)
    wire = fused(g.GEMMAR_FP8_WIRE)
    assert torch.equal(bits(wire), bits(y)), f"{what}: fp8 wire != codec of the band path"
    wire_q = fused(g.GEMMAR_FP8_WIRE | g.GEMMAR_FUSE_QUANTIZE)
    assert torch.equal(bits(wire_q), bits(y)), f"{what}: folded-quantiser wire != codec of the band path"


def draw_gemm_shapes(kind, n, seed):
    rng = np.random.RandomState(seed)
    n_choices = [c for c in range(128, MAX_N + 1, 32) if c % 128 == 0 or (kind == 1 and c % 224 == 0)]
    return [(int(rng.randint(1, MAX_M + 1)), int(rng.choice(n_choices)), int(rng.choice([128, 256, 384, 512])))
            for _ in range(n)]


GEMM_CASES = [(kind, *shape) for kind in (0, 1, 2) for shape in draw_gemm_shapes(kind, 10, 7200 + kind)]


@pytest.mark.parametrize("kind,M,N,K", GEMM_CASES, ids=[f"k{k}-M{M}-N{N}-K{K}" for k, M, N, K in GEMM_CASES])
def test_random_single_gemm(g, ctx, kind, M, N, K):
    make = (blockscale_operands, mx_operands, ptpc_operands)[kind]
    gemm = (g.gemm_blockscale_fp8, g.gemm_mxfp8, g.gemm_ptpc_fp8)[kind]
    A, sa, B, sb = make(1, M, N, K, seed=M * 7 + N * 3 + K)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    gemm(ctx, dev(A[0]), dev(sa[0]), dev(B[0]), dev(sb[0]), C)
    torch.cuda.synchronize()
    assert g.gemmar_status(ctx)[0] == 0
    ref, _ = oracle.gemm_reduce(A, sa, B, sb, kind)
    check_f32_output(C.cpu().numpy(), ref, f"kind {kind} {M}x{N}x{K}")


def draw_reduce_shapes(n, seed):
    rng = np.random.RandomState(seed)
    out = []
    for _ in range(n):
        bands = int(rng.randint(1, 9))
        out.append((int(rng.randint(1, MAX_P + 1)), bands * int(rng.randint(1, 300)),
                    8 * int(rng.randint(1, 257)), bands))
    return out


REDUCE_CASES = draw_reduce_shapes(16, 7300)


@pytest.mark.parametrize("P,M,N,bands", REDUCE_CASES, ids=[f"P{P}-M{M}-N{N}-b{b}" for P, M, N, b in REDUCE_CASES])
def test_random_band_reduce(g, ctx, P, M, N, bands):
    rpb = M // bands
    W = synthetic.normal(P + M + N, synthetic.TID_W, P, (bands, P, rpb, N))
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.band_reduce(ctx, dev(W), P, M, N, bands, out)
    torch.cuda.synchronize()
    assert g.gemmar_status(ctx)[0] == 0
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(bands):
        assert np.array_equal(got[b * rpb:(b + 1) * rpb], oracle.reduce_f32_ordered(W[b])), f"band {b}"


def draw_codec_shapes(n, seed):
    rng = np.random.RandomState(seed)
    return [(int(rng.randint(1, 600)), 16 * int(rng.randint(1, 600)), float(10.0 ** rng.uniform(-20, 20)),
             bool(rng.rand() < 0.5)) for _ in range(n)]


CODEC_CASES = draw_codec_shapes(16, 7400)


@pytest.mark.parametrize("M,N,sigma,bf16", CODEC_CASES,
                         ids=[f"M{M}-N{N}-s{sigma:.0e}-{'bf16' if b else 'f32'}" for M, N, sigma, b in CODEC_CASES])
def test_random_row_codec(g, ctx, M, N, sigma, bf16):
    x = synthetic.normal(M + N, synthetic.TID_X, 3, (M, N), sigma=sigma)
    if bf16:
        xt = torch.from_numpy(x).to(torch.bfloat16)
        x = xt.to(torch.float32).numpy()          # the codec sees exactly these values
        xd = xt.cuda()
    else:
        xd = dev(x)
    q = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    s = torch.empty((M,), dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.rowquant_e4m3(ctx, xd, q, s)
    g.rowdequant_e4m3(ctx, q, s, y)
    torch.cuda.synchronize()
    assert g.gemmar_status(ctx)[0] == 0
    q_ref, s_ref = oracle.rowquant(x)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), oracle.rowdequant(q_ref, s_ref))
