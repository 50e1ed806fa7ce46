"""Failure handling through the C ABI, without faulting the GPU: argument,
shape, alignment and workspace errors return at once and launch nothing; a
band that is never signalled (host-set fault flag) makes the reducer's bounded
wait expire, which the status word reports and which disables the context;
the closed-form self-test passes at create time."""
import numpy as np
import pytest
import torch

from helpers import blockscale_operands

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import block_scaled_fp8_gemm_gb300 as g
    return g


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_create_runs_closed_form_self_test(g):
    torch.cuda.set_device(0)
    ctx = g.gemmar_create(0, 512, 512, 256, 2)        # self-test on (blockscale and mx)
    assert g.gemmar_workspace_bytes(ctx) >= 2 * 512 * 512 * 4
    assert g.gemmar_status(ctx) == (0, 0)
    ctx.close()


def test_host_side_errors_launch_nothing(g):
    torch.cuda.set_device(0)
    ctx = g.gemmar_create(0, 256, 512, 256, 2, flags=g.GEMMAR_NO_SELF_TEST)
    A, sa, B, sb = blockscale_operands(2, 256, 512, 256, seed=1)
    dA, dsa, dB, dsb = [dev(a) for a in A], [dev(s) for s in sa], [dev(b) for b in B], [dev(s) for s in sb]
    out = torch.empty((256, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemmarError) as e:     # M not a multiple of the band count
        g.fused_gemm_reduce(ctx, dA, dsa, dB, dsb, out, bands=3)
    assert e.value.code == g.GEMMAR_ERR_SHAPE
    big = [torch.zeros((1024, 256), dtype=torch.uint8, device="cuda")] * 2
    bigs = [torch.ones((1024, 2), dtype=torch.float32, device="cuda")] * 2
    out2 = torch.empty((1024, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemmarError) as e:     # more rows than the workspace was sized for
        g.fused_gemm_reduce(ctx, big, bigs, dB, dsb, out2)
    assert e.value.code == g.GEMMAR_ERR_WORKSPACE
    raw = torch.empty(256 * 512 * 2 + 16, dtype=torch.uint8, device="cuda")
    misaligned = raw[8:8 + 256 * 512 * 2].view(torch.bfloat16).view(256, 512)
    with pytest.raises(g.GemmarError) as e:
        g.fused_gemm_reduce(ctx, dA, dsa, dB, dsb, misaligned)
    assert e.value.code == g.GEMMAR_ERR_ALIGN
    torch.cuda.synchronize()
    assert g.gemmar_status(ctx)[0] == 0
    ctx.close()


def test_empty_inputs_are_refused_before_any_launch(g):
    """Zero rows through every entry point: refused on the host (argument or shape
    error), nothing launched, the context's status clean afterwards."""
    torch.cuda.set_device(0)
    ctx = g.gemmar_create(0, 256, 512, 256, 2, flags=g.GEMMAR_NO_SELF_TEST)
    u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device="cuda")
    f32 = lambda *s: torch.empty(s, dtype=torch.float32, device="cuda")
    bf = lambda *s: torch.empty(s, dtype=torch.bfloat16, device="cuda")
    B, sb = [u8(512, 256)] * 2, [f32(4, 2)] * 2
    calls = {
        "fused_gemm_reduce": lambda: g.fused_gemm_reduce(ctx, [u8(0, 256)] * 2, [f32(0, 2)] * 2, B, sb, bf(0, 512)),
        "gemm_blockscale_fp8": lambda: g.gemm_blockscale_fp8(ctx, u8(0, 256), f32(0, 2), B[0], sb[0], bf(0, 512)),
        "rowquant_e4m3": lambda: g.rowquant_e4m3(ctx, bf(0, 512), u8(0, 512), f32(0)),
        "rowdequant_e4m3": lambda: g.rowdequant_e4m3(ctx, u8(0, 512), f32(0), bf(0, 512)),
        "quant_blockscale_e4m3": lambda: g.quant_blockscale_e4m3(ctx, bf(0, 256), 1, u8(0, 256), f32(0, 2)),
    }
    for name, call in calls.items():
        with pytest.raises(g.GemmarError) as e:
            call()
        assert e.value.code in (g.GEMMAR_ERR_ARG, g.GEMMAR_ERR_SHAPE), (name, e.value.code)
    torch.cuda.synchronize()
    assert g.gemmar_status(ctx) == (0, 0)
    ctx.close()


@pytest.mark.parametrize("kind,create_flags,call_flags",
                         [(0, 0, 0), (0, "pair", 0), (1, 0, 0), (2, 0, 0), (0, 0, "fuse_quantize")],
                         ids=["blockscale", "blockscale-cta-pair", "mx", "ptpc", "blockscale-fused-quantize"])
def test_unsignalled_band_times_out_cleanly(g, kind, create_flags, call_flags):
    from helpers import mx_operands, ptpc_operands
    torch.cuda.set_device(0)
    cflags = g.GEMMAR_NO_SELF_TEST | (g.GEMMAR_CTA_PAIR if create_flags == "pair" else 0)
    ctx = g.gemmar_create(0, 256, 512, 256, 2, flags=cflags, wait_timeout_ns=50_000_000)
    make = {0: blockscale_operands, 1: mx_operands, 2: ptpc_operands}[kind]
    A, sa, B, sb = make(2, 256, 512, 256, seed=2)
    dA, dsa, dB, dsb = [dev(a) for a in A], [dev(s) for s in sa], [dev(b) for b in B], [dev(s) for s in sb]
    out = torch.empty((256, 512), dtype=torch.bfloat16, device="cuda")
    extra = g.GEMMAR_FP8_WIRE | g.GEMMAR_FUSE_QUANTIZE if call_flags == "fuse_quantize" else 0
    g.fused_gemm_reduce(ctx, dA, dsa, dB, dsb, out, scale_kind=kind, flags=g.GEMMAR_FAULT_SKIP_BAND | extra)
    torch.cuda.synchronize()                    # the wait gave up: no hang, context still usable
    code, detail = g.gemmar_status(ctx)
    assert code == g.GEMMAR_ERR_TIMEOUT and detail == 7      # the reducer's band wait
    with pytest.raises(g.GemmarError) as e:     # sticky-disabled afterwards
        g.fused_gemm_reduce(ctx, dA, dsa, dB, dsb, out, scale_kind=kind)
    assert e.value.code == g.GEMMAR_ERR_DISABLED
    ctx.close()
    # a fresh context on the same device works
    ctx2 = g.gemmar_create(0, 256, 512, 256, 2, flags=cflags)
    g.fused_gemm_reduce(ctx2, dA, dsa, dB, dsb, out, scale_kind=kind)
    torch.cuda.synchronize()
    assert g.gemmar_status(ctx2)[0] == 0
    ctx2.close()
