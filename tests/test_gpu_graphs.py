"""The fused path captured in a CUDA graph and replayed: every step of it is a
stream-ordered launch or memset on the caller's stream, so a captured call
replays the same work on whatever the input buffers hold at replay time.
Checked bit for bit against eager calls, for the band path with its in-kernel
reduce, the fp8 wire, mxfp8, and the allocation-free entry point."""
import numpy as np
import pytest
import torch

from helpers import blockscale_operands, mx_operands

pytestmark = pytest.mark.gpu

P, M, N, K, BANDS = 8, 1024, 1024, 512, 8


@pytest.fixture(scope="module")
def g():
    import block_scaled_fp8_gemm_gb300 as g
    return g


@pytest.fixture(scope="module")
def ctx(g):
    torch.cuda.set_device(0)
    c = g.gemmar_create(0, M, N, K, P, flags=g.GEMMAR_NO_SELF_TEST, wait_timeout_ns=1_000_000_000)
    yield c
    c.close()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def capture(fn):
    """Capture fn() on a side stream after one warm-up call there."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


@pytest.mark.parametrize("kind,flags", [(0, 0), (0, 1), (1, 0), (0, 128)])
def test_graph_replay_equals_eager(g, ctx, kind, flags):
    make = blockscale_operands if kind == 0 else mx_operands
    A, sa, B, sb = [[dev(x) for x in xs] for xs in make(P, M, N, K, seed=21)]
    eager = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.fused_gemm_reduce(ctx, A, sa, B, sb, eager, scale_kind=kind, bands=BANDS, flags=flags)
    torch.cuda.synchronize()
    assert g.gemmar_status(ctx)[0] == 0

    out = torch.empty_like(eager)
    graph = capture(lambda: g.fused_gemm_reduce(ctx, A, sa, B, sb, out, scale_kind=kind, bands=BANDS, flags=flags))
    out.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert g.gemmar_status(ctx)[0] == 0
    assert same(out, eager)

    # new contents in the same buffers: the replay reads them
    A2, sa2, _, _ = make(P, M, N, K, seed=22)
    for d, h in zip(A + sa, A2 + sa2):
        d.copy_(torch.from_numpy(np.ascontiguousarray(h)))
    graph.replay()
    ref2 = torch.empty_like(eager)
    g.fused_gemm_reduce(ctx, A, sa, B, sb, ref2, scale_kind=kind, bands=BANDS, flags=flags)
    torch.cuda.synchronize()
    assert g.gemmar_status(ctx)[0] == 0
    assert same(out, ref2)
    assert not same(ref2, eager)


def test_graph_replay_noalloc(g):
    torch.cuda.set_device(0)
    A, sa, B, sb = [[dev(x) for x in xs] for xs in blockscale_operands(P, M, N, K, seed=23)]
    eager = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.fused_gemm_reduce_noalloc(A, sa, B, sb, eager, bands=BANDS)
    torch.cuda.synchronize()
    out = torch.empty_like(eager)
    graph = capture(lambda: g.fused_gemm_reduce_noalloc(A, sa, B, sb, out, bands=BANDS))
    out.zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert same(out, eager)
