"""GPU parity of the streaming kernels against the oracle, through the C ABI:
the per-row e4m3 codec (bit-exact), the device quantisers (bit-exact) and the
fixed-order band reduce (bit-exact against the ordered fp32 definition, and
within tolerance of the fp64 oracle)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from helpers import check_bf16_output, rel_l2

pytestmark = pytest.mark.gpu

TABLE = oracle.e4m3_decode_table()


@pytest.fixture(scope="module")
def g():
    import block_scaled_fp8_gemm_gb300 as g
    return g


@pytest.fixture(scope="module")
def ctx(g):
    torch.cuda.set_device(0)
    c = g.gemmar_create(0, 512, 256, 128, 2, flags=g.GEMMAR_NO_SELF_TEST, wait_timeout_ns=500_000_000)
    yield c
    c.close()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_status_ok(g, ctx):
    torch.cuda.synchronize()
    code, detail = g.gemmar_status(ctx)
    assert code == 0, (code, detail)


# ---------------------------------------------------------------- row codec

def codec_gpu(g, ctx, x_t):
    M, N = x_t.shape
    q = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    s = torch.empty((M,), dtype=torch.float32, device="cuda")
    g.rowquant_e4m3(ctx, x_t, q, s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.rowdequant_e4m3(ctx, q, s, y)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy(), u16(y)


def test_rowcodec_bitexact_fp32_page_payload(g, ctx):
    # the page's payload shape: [2048, 7168] standard normal, fed as identical fp32 rows
    x = synthetic.normal(0, synthetic.TID_X, 0, (2048, 7168))
    q, s, y = codec_gpu(g, ctx, dev(x))
    q_ref, s_ref = oracle.rowquant(x)
    assert np.array_equal(s, s_ref)
    assert np.array_equal(q, q_ref)
    assert np.array_equal(y, oracle.rowdequant(q_ref, s_ref))
    err = rel_l2(oracle.bf16_to_f32(y), x)
    assert abs(err - 2.646e-2) < 0.01 * 2.646e-2      # the page's per-row figure


def test_rowcodec_bitexact_bf16_rows(g, ctx):
    x32 = synthetic.normal(1, synthetic.TID_X, 1, (333, 7168), sigma=3.0)
    xb = torch.from_numpy(x32).to(torch.bfloat16)
    x_exact = xb.to(torch.float32).numpy()             # bf16 -> fp32 is exact
    q, s, y = codec_gpu(g, ctx, xb.cuda())
    q_ref, s_ref = oracle.rowquant(x_exact)
    assert np.array_equal(s, s_ref) and np.array_equal(q, q_ref)
    assert np.array_equal(y, oracle.rowdequant(q_ref, s_ref))


def test_rowcodec_edge_cases(g, ctx):
    x = synthetic.normal(2, synthetic.TID_X, 2, (8, 256))
    x[0] = 0.0                                       # zero row
    x[1] = -0.0                                      # negative-zero row
    x[2, 5] = 448.0 * 16                             # amax a power of two of 448
    x[3] = np.float32(2.0 ** -118) * x[3]            # tiny row (subnormal codes)
    x[4, ::2] = 0.0                                  # zeros inside a row
    x[5] *= np.float32(1e30)                         # huge row
    x[6, 100] = -x[6].__abs__().max() * 2            # negative amax
    for M in (8, 3, 1):                              # ragged row counts
        q, s, y = codec_gpu(g, ctx, dev(x[:M]))
        q_ref, s_ref = oracle.rowquant(x[:M])
        assert np.array_equal(s, s_ref) and np.array_equal(q, q_ref)
        assert np.array_equal(y, oracle.rowdequant(q_ref, s_ref))


def _nan_as_one(codes):
    """e4m3 codes with both NaN codes (0x7F, 0xFF) mapped to 0x7F: the sign of a
    NaN is not something the encoding fixes."""
    c = np.asarray(codes, dtype=np.uint8).copy()
    c[(c & 0x7F) == 0x7F] = 0x7F
    return c


def _non_finite_rows(C):
    x = synthetic.normal(5, synthetic.TID_X, 5, (6, C))
    x[0, 7] = np.inf                                 # one +inf: scale inf, the rest +-0 codes, inf -> NaN
    x[1, 9] = -np.inf
    x[2, 11] = np.nan                                # a NaN is skipped by the amax, coded NaN
    x[3] = np.nan                                    # all NaN: amax 0, scale 0, +0 codes
    x[4, 3], x[4, C - 1] = np.inf, -np.inf
    return x                                         # row 5: finite control


@pytest.mark.parametrize("C", [256, 1024])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_quantisers_with_non_finite_inputs(g, ctx, dtype, C):
    """Infinities and NaN in the quantised rows (an overflowing layer): the row
    codec's and the 1x128 and mx quantisers' codes and scales match the oracle,
    the two NaN codes taken as one.  bf16 rows of 1024 take the single-pass row
    quantiser, whose amax runs on packed bf16 pairs."""
    xd, xw = _as_input(_non_finite_rows(C), dtype)
    q = torch.empty((6, C), dtype=torch.uint8, device="cuda")
    s = torch.empty((6,), dtype=torch.float32, device="cuda")
    g.rowquant_e4m3(ctx, xd, q, s)
    sg = torch.empty((6, C // 128), dtype=torch.float32, device="cuda")
    qg = torch.empty((6, C), dtype=torch.uint8, device="cuda")
    g.quant_blockscale_e4m3(ctx, xd, 1, qg, sg)
    em = torch.empty((6, C // 32), dtype=torch.uint8, device="cuda")
    qm = torch.empty((6, C), dtype=torch.uint8, device="cuda")
    g.quant_mx_e4m3(ctx, xd, qm, em)
    assert_status_ok(g, ctx)
    q_ref, s_ref = oracle.rowquant(xw)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(_nan_as_one(q.cpu().numpy()), _nan_as_one(q_ref))
    qg_ref, sg_ref = oracle.quant_block(xw, 1, 128)
    assert np.array_equal(sg.cpu().numpy(), sg_ref)
    assert np.array_equal(_nan_as_one(qg.cpu().numpy()), _nan_as_one(qg_ref))
    qm_ref, em_ref = oracle.quant_mx(xw)
    assert np.array_equal(em.cpu().numpy(), em_ref)
    assert np.array_equal(_nan_as_one(qm.cpu().numpy()), _nan_as_one(qm_ref))


def test_rowdequant_all_codes(g, ctx):
    codes = np.arange(256, dtype=np.uint8)
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    q = np.tile(codes, (6, 1))
    s = np.array([1.0, 0.5, 3.0, 1e-30, 7e30, 0.0], dtype=np.float32)
    y = torch.empty((6, 256), dtype=torch.bfloat16, device="cuda")
    g.rowdequant_e4m3(ctx, dev(q), dev(s), y)
    torch.cuda.synchronize()
    assert np.array_equal(u16(y), oracle.rowdequant(q, s))


# ---------------------------------------------------------------- quantisers

def _as_input(x, dtype):
    """The quantiser's device input of dtype, and its exact fp32 value (bf16
    widens to fp32 exactly) for the oracle."""
    xt = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    return xt.cuda(), xt.float().numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("R,C,gr", [(256, 512, 1), (77, 384, 1), (3, 128, 1), (256, 512, 128), (300, 256, 128),
                                    (5, 384, 128)])
def test_quant_blockscale_bitexact(g, ctx, R, C, gr, dtype):
    x = synthetic.normal(3, synthetic.TID_A, R, (R, C), sigma=0.02 if gr == 128 else 1.0)
    x[0, :128] = 0.0
    x[-1, -128:] = np.float32(448.0 * 2.0 ** -7)     # a group whose amax is a power of two of 448
    xd, xw = _as_input(x, dtype)
    q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    s = torch.empty(((R + gr - 1) // gr, C // 128), dtype=torch.float32, device="cuda")
    g.quant_blockscale_e4m3(ctx, xd, gr, q, s)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_block(xw, gr, 128)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("R,C", [(128, 256), (37, 96), (3, 32)])
def test_quant_mx_bitexact(g, ctx, R, C, dtype):
    x = synthetic.normal(4, synthetic.TID_A, R, (R, C))
    x[1 % R, 0:32] = 0.0
    x[2 % R, C - 32:C] = np.float32(448.0 * 2.0 ** -5)       # a group on an exact power of two of 448
    x[R - 1, 0:32] *= np.float32(2.0 ** -100)
    xd, xw = _as_input(x, dtype)
    q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    e = torch.empty((R, C // 32), dtype=torch.uint8, device="cuda")
    g.quant_mx_e4m3(ctx, xd, q, e)
    torch.cuda.synchronize()
    q_ref, e_ref = oracle.quant_mx(xw)
    assert np.array_equal(e.cpu().numpy(), e_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quant_blockscale_bf16_wo_b_activation(g, ctx):
    """The call site's own case: wo_b's bf16 activations [4096, 2048] quantised
    per 1x128 on the device, bit for bit against the oracle quantiser fed the
    same rows."""
    x = synthetic.normal(6, synthetic.TID_A, 0, (4096, 2048))
    xd, xw = _as_input(x, "bf16")
    q = torch.empty((4096, 2048), dtype=torch.uint8, device="cuda")
    s = torch.empty((4096, 16), dtype=torch.float32, device="cuda")
    g.quant_blockscale_e4m3(ctx, xd, 1, q, s)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_act_1x128(xw)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def _amax_sweep_bits(C=2048):
    """bf16 bit patterns [R, C]: every 128-wide group starts with its amax, taken
    over all 128 bf16 significands at exponents from -122 (amax / 448 below the
    smallest scale the encoder's guarded products take, down to subnormal
    scales) to 127, followed by
    seeded bf16 patterns at or below it with alternating signs (subnormal bf16
    included).  Exact e4m3 midpoints of x / s occur for every amax significand."""
    exps = np.array(list(range(-122, -100)) + list(range(-20, 20, 3)) + list(range(100, 128)))
    amax = (((exps[:, None] + 127) << 7) | (np.arange(128)[None, :])).reshape(-1).astype(np.uint32)
    rng = np.random.default_rng(11)
    body = np.floor(rng.random((amax.size, 127)) * (amax[:, None] + 1)).astype(np.uint32)
    body |= (np.arange(127, dtype=np.uint32) % 2)[None, :] << 15
    bits = np.concatenate([amax[:, None], body], axis=1).astype(np.uint16)
    return bits.reshape(-1, C)


def test_quantisers_over_an_amax_sweep(g, ctx):
    """The 1x128, row and mx quantisers on bf16 rows whose groups' amax runs over
    every significand and exponent: codes and scales bit for bit against the
    oracle (the guarded encoder's fast path, its division fallback at exact
    midpoints and its exact path below the smallest scale)."""
    bits = _amax_sweep_bits()
    R, C = bits.shape
    xd = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    xw = xd.float().cpu().numpy()
    q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    s = torch.empty((R, C // 128), dtype=torch.float32, device="cuda")
    g.quant_blockscale_e4m3(ctx, xd, 1, q, s)
    qm = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    em = torch.empty((R, C // 32), dtype=torch.uint8, device="cuda")
    g.quant_mx_e4m3(ctx, xd, qm, em)
    qr, sr, _ = codec_gpu(g, ctx, xd)
    assert_status_ok(g, ctx)
    q_ref, s_ref = oracle.quant_block(xw, 1, 128)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    qm_ref, em_ref = oracle.quant_mx(xw)
    assert np.array_equal(em.cpu().numpy(), em_ref) and np.array_equal(qm.cpu().numpy(), qm_ref)
    qr_ref, sr_ref = oracle.rowquant(xw)
    assert np.array_equal(sr, sr_ref) and np.array_equal(qr, qr_ref)


# ---------------------------------------------------------------- band reduce

@pytest.mark.parametrize("P,M,N,bands", [(2, 256, 512, 2), (8, 512, 256, 8), (1, 128, 128, 1),
                                         (3, 96, 384, 3), (5, 40, 128, 5), (8, 512, 256, 1)])
def test_band_reduce_bitexact(g, ctx, P, M, N, bands):
    rpb = M // bands
    W = synthetic.normal(5, synthetic.TID_W, P, (bands, P, rpb, N))
    W[..., 0] = np.float32(1e-30)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.band_reduce(ctx, dev(W), P, M, N, bands, out)
    torch.cuda.synchronize()
    got = u16(out)
    for b in range(bands):
        ref = oracle.reduce_f32_ordered(W[b])
        assert np.array_equal(got[b * rpb:(b + 1) * rpb], ref), f"band {b}"
    # and within the tolerance of the fp64 sum
    exact = W.astype(np.float64).sum(axis=1).reshape(M, N)
    check_bf16_output(oracle.bf16_to_f32(got), exact, "band_reduce vs fp64")
