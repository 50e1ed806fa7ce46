"""The allocation-free entry point (fused_gemm_reduce_noalloc), for callers
that cannot call cudaMalloc -- e.g. engines that own all device memory in a
pool of their own.  Called through the C ABI and checked against the existing
fused_gemm_reduce on the same inputs, twice in a row (the fixed scratch keeps
the previous call's contents, so the second call checks that it starts
clean); its status read-back reports a clean run, and a call after the first
changes neither the device's free memory nor torch's allocations.  Collected
last, so a stop-at-first-failure run has already run every other test."""
import gc

import numpy as np
import pytest
import torch

import oracle
from helpers import blockscale_operands, check_bf16_output

pytestmark = pytest.mark.gpu


def test_noalloc_matches_fused_twice():
    import block_scaled_fp8_gemm_gb300 as g
    torch.cuda.set_device(0)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ctx = g.gemmar_create(0, 512, 512, 256, 4, flags=g.GEMMAR_NO_SELF_TEST)
    try:
        for seed, (P, M, N, K, bands) in enumerate([(2, 256, 512, 256, 2), (4, 512, 384, 256, 4)]):
            A, sa, B, sb = blockscale_operands(P, M, N, K, seed=40 + seed)
            dA, dsa, dB, dsb = [dev(a) for a in A], [dev(s) for s in sa], [dev(b) for b in B], [dev(s) for s in sb]
            ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            g.fused_gemm_reduce(ctx, dA, dsa, dB, dsb, ref, bands=bands)
            got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            g.fused_gemm_reduce_noalloc(dA, dsa, dB, dsb, got, bands=bands)
            torch.cuda.synchronize()
            assert g.gemmar_status(ctx)[0] == 0
            assert g.fused_gemm_reduce_noalloc_status() == (0, 0)
            r = ref.float().cpu().numpy()
            # within the tolerance the parity tests use (and in fact bit for bit)
            check_bf16_output(got.float().cpu().numpy(), r, f"noalloc vs fused, call {seed}")
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
            exact, _ = oracle.gemm_reduce(A, sa, B, sb, 0)
            check_bf16_output(got.float().cpu().numpy(), exact, f"noalloc vs oracle, call {seed}")
    finally:
        ctx.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import block_scaled_fp8_gemm_gb300 as g
    torch.cuda.set_device(0)
    P, M, N, K = 8, 2048, 1024, 128          # 16 M partials > the 8 M the scratch holds
    assert P * M * N > g.GEMMAR_NOALLOC_MAX_PARTIALS
    A = [torch.zeros((M, K), dtype=torch.uint8, device="cuda")] * P
    sa = [torch.ones((M, 1), dtype=torch.float32, device="cuda")] * P
    B = [torch.zeros((N, K), dtype=torch.uint8, device="cuda")] * P
    sb = [torch.ones((N // 128, 1), dtype=torch.float32, device="cuda")] * P
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemmarError) as e:
        g.fused_gemm_reduce_noalloc(A, sa, B, sb, out)
    assert e.value.code == g.GEMMAR_ERR_WORKSPACE


def test_noalloc_allocates_nothing():
    """After a first call (which looks up the scratch), further calls leave the
    device's free memory and torch's allocated bytes unchanged."""
    import block_scaled_fp8_gemm_gb300 as g
    torch.cuda.set_device(0)
    P, M, N, K = 4, 512, 512, 256
    A, sa, B, sb = blockscale_operands(P, M, N, K, seed=77)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    dA, dsa, dB, dsb = [dev(a) for a in A], [dev(s) for s in sa], [dev(b) for b in B], [dev(s) for s in sb]
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.fused_gemm_reduce_noalloc(dA, dsa, dB, dsb, out)
    torch.cuda.synchronize()
    first = out.clone()
    gc.collect()   # tensors of earlier tests released now, not between the two readings
    torch.cuda.synchronize()
    free0, allocated0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(2):
        g.fused_gemm_reduce_noalloc(dA, dsa, dB, dsb, out)
    torch.cuda.synchronize()
    free1, allocated1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    assert g.fused_gemm_reduce_noalloc_status() == (0, 0)
    assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert allocated1 == allocated0
