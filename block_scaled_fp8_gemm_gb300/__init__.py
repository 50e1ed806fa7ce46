"""block_scaled_fp8_gemm_gb300 -- Python binding of libgemmar (include/gemmar.h).

The wo_b path of a DeepSeek-style attention block on one GB300: block-scaled
e4m3 GEMMs per K-slice (tcgen05 MMA, TMEM accumulators, TMA-fed shared
stages), the fixed-order fp32 band reduce to bf16, the per-row e4m3 "fp8 wire"
codec, and the mxfp8 variant on the native block-scaled MMA.

Every function here has the name of the C entry point it calls and only
marshals arguments: torch tensors supply device memory, torch streams supply
the CUDA stream, and all arithmetic runs in the library's CUDA kernels.  The
library is required: importing this package raises if ``libgemmar.so`` has not
been built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgemmar.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libgemmar.so not found at {LIB_PATH}; build it first with "
        "block_scaled_fp8_gemm_gb300.build.build() (there is no fallback path)")

_lib = ctypes.CDLL(LIB_PATH)

# ---- constants (mirror include/gemmar.h) -------------------------------------
GEMMAR_OK = 0
GEMMAR_ERR_ARG = 1
GEMMAR_ERR_SHAPE = 2
GEMMAR_ERR_ALIGN = 3
GEMMAR_ERR_WORKSPACE = 4
GEMMAR_ERR_CUDA = 5
GEMMAR_ERR_TIMEOUT = 6
GEMMAR_ERR_DISABLED = 7
GEMMAR_ERR_DEVICE = 8
STATUS_NAMES = {0: "OK", 1: "ERR_ARG", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_WORKSPACE",
                5: "ERR_CUDA", 6: "ERR_TIMEOUT", 7: "ERR_DISABLED", 8: "ERR_DEVICE"}

GEMMAR_DTYPE_F32 = 0
GEMMAR_DTYPE_BF16 = 1
GEMMAR_SCALE_BLOCK128 = 0
GEMMAR_SCALE_MX32 = 1
GEMMAR_SCALE_PTPC = 2
GEMMAR_FP8_WIRE = 1 << 0
GEMMAR_DEBUG_CANARY = 1 << 1
GEMMAR_FAULT_SKIP_BAND = 1 << 2
GEMMAR_NO_SELF_TEST = 1 << 3
GEMMAR_FUSE_SLICES = 1 << 4
GEMMAR_CTA_PAIR = 1 << 5
GEMMAR_FUSE_ONCHIP = 1 << 6
GEMMAR_SERIAL_REDUCE = 1 << 7
GEMMAR_FUSE_QUANTIZE = 1 << 8
GEMMAR_MAX_P = 8
GEMMAR_NOALLOC_MAX_PARTIALS = 8 * 1024 * 1024

# ---- signatures ----------------------------------------------------------------
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_U32 = ctypes.c_uint32
_PP = ctypes.POINTER(ctypes.c_void_p)

_SIGS = {
    "gemmar_supports": (_I, [_I, _I64, _I64, _I64, _I, _I]),
    "gemmar_create": (_I, [ctypes.POINTER(_P), _I, _I64, _I64, _I64, _I, _U32, _I64]),
    "gemmar_destroy": (_I, [_P]),
    "gemmar_status": (_I, [_P, ctypes.POINTER(_I)]),
    "gemmar_workspace_bytes": (_I64, [_P]),
    "gemmar_set_phase_timing": (_I, [_P, _I]),
    "gemmar_phase_times": (_I, [_P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(_I)]),
    "gemmar_overlap_stats": (_I, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "gemm_blockscale_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P]),
    "gemm_mxfp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P]),
    "gemm_ptpc_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P]),
    "band_reduce": (_I, [_P, _P, _I, _I64, _I64, _I, _P, _P]),
    "rowquant_e4m3": (_I, [_P, _P, _I, _I64, _I64, _P, _P, _P]),
    "rowdequant_e4m3": (_I, [_P, _P, _P, _I64, _I64, _P, _P]),
    "quant_blockscale_e4m3": (_I, [_P, _P, _I, _I64, _I64, _I, _P, _P, _P]),
    "quant_mx_e4m3": (_I, [_P, _P, _I, _I64, _I64, _P, _P, _P]),
    "fused_gemm_reduce": (_I, [_P, _I, _PP, _PP, _PP, _PP, _I, _I64, _I64, _I64, _I, _U32, _P, _P]),
    "fused_gemm_reduce_noalloc": (_I, [_I, _PP, _PP, _PP, _PP, _I64, _I64, _I64, _I, _P, _P]),
    "fused_gemm_reduce_noalloc_status": (_I, [ctypes.POINTER(_I)]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


class GemmarError(RuntimeError):
    def __init__(self, code: int, where: str, detail: int = 0):
        self.code = code
        self.detail = detail
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} (code {code}, detail {detail})")


def _check(code: int, where: str):
    if code != GEMMAR_OK:
        raise GemmarError(code, where)


def _ptr(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _u8(t: torch.Tensor, name: str) -> int:
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"{name} must be uint8 codes (or float8_e4m3fn), got {t.dtype}")
    return _ptr(t, name)


def _f32(t: torch.Tensor, name: str) -> int:
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    return _ptr(t, name)


def _bf16(t: torch.Tensor, name: str) -> int:
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    return _ptr(t, name)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class Context:
    """Owns one gemmar_ctx (its workspace and status word)."""

    def __init__(self, handle: int, device: int):
        self._h = ctypes.c_void_p(handle)
        self.device = device

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise ValueError("context already destroyed")
        return self._h

    def close(self):
        if self._h:
            with torch.cuda.device(self.device):
                gemmar_destroy(self)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- entry points ------------------------------------------------------------------

def gemmar_supports(P: int, M: int, N: int, K: int, bands: int = 0,
                    scale_kind: int = GEMMAR_SCALE_BLOCK128) -> int:
    return int(_lib.gemmar_supports(P, M, N, K, bands if bands else P, scale_kind))


def gemmar_create(device: int, max_M: int, N: int, K: int, max_P: int, flags: int = 0,
                  wait_timeout_ns: int = 0) -> Context:
    h = ctypes.c_void_p()
    with torch.cuda.device(device):
        _check(_lib.gemmar_create(ctypes.byref(h), device, max_M, N, K, max_P, flags, wait_timeout_ns),
               "gemmar_create")
    return Context(h.value, device)


def gemmar_destroy(ctx: Context) -> None:
    h = ctx._h
    ctx._h = ctypes.c_void_p()
    if h:
        _check(_lib.gemmar_destroy(h), "gemmar_destroy")


def gemmar_status(ctx: Context):
    """(code, detail) of the device status word; call after the work completed."""
    d = ctypes.c_int(0)
    code = int(_lib.gemmar_status(ctx.handle, ctypes.byref(d)))
    return code, int(d.value)


def gemmar_workspace_bytes(ctx: Context) -> int:
    return int(_lib.gemmar_workspace_bytes(ctx.handle))


GEMMAR_NUM_PHASES = 4
PHASE_NAMES = ("gemm", "reduce", "quantize", "dequantize")


def gemmar_set_phase_timing(ctx: Context, enable: bool = True) -> None:
    _check(_lib.gemmar_set_phase_timing(ctx.handle, 1 if enable else 0), "gemmar_set_phase_timing")


def gemmar_phase_times(ctx: Context):
    """(dict phase -> summed ms, number of recorded calls); clears the record."""
    ms = (ctypes.c_float * GEMMAR_NUM_PHASES)()
    calls = ctypes.c_int(0)
    _check(_lib.gemmar_phase_times(ctx.handle, ms, ctypes.byref(calls)), "gemmar_phase_times")
    return {PHASE_NAMES[i]: float(ms[i]) for i in range(GEMMAR_NUM_PHASES)}, int(calls.value)


def gemmar_overlap_stats(ctx: Context):
    """(blocks summed by the GEMM kernel while it ran, all 32 x 32 output blocks)
    of the last fused band-path call; call after its work completed."""
    ov = ctypes.c_int64(0)
    tot = ctypes.c_int64(0)
    _check(_lib.gemmar_overlap_stats(ctx.handle, ctypes.byref(ov), ctypes.byref(tot)), "gemmar_overlap_stats")
    return int(ov.value), int(tot.value)


def _cdtype(C: torch.Tensor) -> int:
    if C.dtype == torch.float32:
        return GEMMAR_DTYPE_F32
    if C.dtype == torch.bfloat16:
        return GEMMAR_DTYPE_BF16
    raise TypeError(f"C must be float32 or bfloat16, got {C.dtype}")


def gemm_blockscale_fp8(ctx: Context, A, sa, B, sb, C, stream=None) -> None:
    M, K = A.shape
    N = B.shape[0]
    _check(_lib.gemm_blockscale_fp8(ctx.handle, _u8(A, "A"), _f32(sa, "sa"), _u8(B, "B"), _f32(sb, "sb"),
                                    _ptr(C, "C"), _cdtype(C), M, N, K, _stream(stream)),
           "gemm_blockscale_fp8")


def gemm_ptpc_fp8(ctx: Context, A, sa, B, sb, C, stream=None) -> None:
    """C = (sa[m]*sb[n]) * A @ B^T with per-token sa [M] and per-channel sb [N] (fp32)."""
    M, K = A.shape
    N = B.shape[0]
    _check(_lib.gemm_ptpc_fp8(ctx.handle, _u8(A, "A"), _f32(sa, "sa"), _u8(B, "B"), _f32(sb, "sb"),
                              _ptr(C, "C"), _cdtype(C), M, N, K, _stream(stream)),
           "gemm_ptpc_fp8")


def gemm_mxfp8(ctx: Context, A, ea, B, eb, C, stream=None) -> None:
    M, K = A.shape
    N = B.shape[0]
    _check(_lib.gemm_mxfp8(ctx.handle, _u8(A, "A"), _u8(ea, "ea"), _u8(B, "B"), _u8(eb, "eb"),
                           _ptr(C, "C"), _cdtype(C), M, N, K, _stream(stream)),
           "gemm_mxfp8")


def band_reduce(ctx: Context, W, P: int, M: int, N: int, bands: int, out, stream=None) -> None:
    _check(_lib.band_reduce(ctx.handle, _f32(W, "W"), P, M, N, bands, _bf16(out, "out"), _stream(stream)),
           "band_reduce")


def _xdtype(x) -> int:
    if x.dtype == torch.bfloat16:
        return GEMMAR_DTYPE_BF16
    if x.dtype == torch.float32:
        return GEMMAR_DTYPE_F32
    raise TypeError(f"x must be bfloat16 or float32, got {x.dtype}")


def rowquant_e4m3(ctx: Context, x, q, row_scale, stream=None) -> None:
    M, N = x.shape
    _check(_lib.rowquant_e4m3(ctx.handle, _ptr(x, "x"), _xdtype(x), M, N, _u8(q, "q"),
                              _f32(row_scale, "row_scale"), _stream(stream)),
           "rowquant_e4m3")


def rowdequant_e4m3(ctx: Context, q, row_scale, y, stream=None) -> None:
    M, N = q.shape
    _check(_lib.rowdequant_e4m3(ctx.handle, _u8(q, "q"), _f32(row_scale, "row_scale"), M, N, _bf16(y, "y"),
                                _stream(stream)),
           "rowdequant_e4m3")


def quant_blockscale_e4m3(ctx: Context, x, group_rows: int, q, scales, stream=None) -> None:
    """Blockscale quantiser of a bf16 or fp32 [R, C] matrix (group_rows 1 or 128)."""
    R, C = x.shape
    _check(_lib.quant_blockscale_e4m3(ctx.handle, _ptr(x, "x"), _xdtype(x), R, C, group_rows, _u8(q, "q"),
                                      _f32(scales, "scales"), _stream(stream)),
           "quant_blockscale_e4m3")


def quant_mx_e4m3(ctx: Context, x, q, e8m0, stream=None) -> None:
    """mxfp8 quantiser (ue8m0 per 1x32) of a bf16 or fp32 [R, C] matrix."""
    R, C = x.shape
    _check(_lib.quant_mx_e4m3(ctx.handle, _ptr(x, "x"), _xdtype(x), R, C, _u8(q, "q"), _u8(e8m0, "e8m0"),
                              _stream(stream)),
           "quant_mx_e4m3")


def fused_gemm_reduce(ctx: Context, A: Sequence, sa: Sequence, B: Sequence, sb: Sequence, out,
                      scale_kind: int = GEMMAR_SCALE_BLOCK128, bands: int = 0, flags: int = 0,
                      stream=None) -> None:
    P = len(A)
    if not (len(sa) == len(B) == len(sb) == P):
        raise ValueError("A, sa, B, sb must have one entry per slice")
    M, K = A[0].shape
    N = B[0].shape[0]
    sc = _u8 if scale_kind == GEMMAR_SCALE_MX32 else _f32
    arr = lambda ptrs: (ctypes.c_void_p * P)(*ptrs)
    pa = arr([_u8(a, "A[p]") for a in A])
    pb = arr([_u8(b, "B[p]") for b in B])
    psa = arr([sc(s, "sa[p]") for s in sa])
    psb = arr([sc(s, "sb[p]") for s in sb])
    cast = lambda x: ctypes.cast(x, _PP)
    _check(_lib.fused_gemm_reduce(ctx.handle, P, cast(pa), cast(psa), cast(pb), cast(psb), scale_kind,
                                  M, N, K, bands, flags, _bf16(out, "out"), _stream(stream)),
           "fused_gemm_reduce")


def fused_gemm_reduce_noalloc(A: Sequence, sa: Sequence, B: Sequence, sb: Sequence, out, bands: int = 0,
                              stream=None) -> None:
    """Blockscale fused GEMM + band reduce that allocates no device memory
    (its scratch is fixed-size library memory, at most
    GEMMAR_NOALLOC_MAX_PARTIALS fp32 partials).  For callers that cannot call
    cudaMalloc, e.g. engines owning all device memory in a pool of their own."""
    P = len(A)
    if not (len(sa) == len(B) == len(sb) == P):
        raise ValueError("A, sa, B, sb must have one entry per slice")
    M, K = A[0].shape
    N = B[0].shape[0]
    arr = lambda ptrs: ctypes.cast((ctypes.c_void_p * P)(*ptrs), _PP)
    _check(_lib.fused_gemm_reduce_noalloc(P, arr([_u8(a, "A[p]") for a in A]), arr([_f32(s, "sa[p]") for s in sa]),
                                          arr([_u8(b, "B[p]") for b in B]), arr([_f32(s, "sb[p]") for s in sb]),
                                          M, N, K, bands, _bf16(out, "out"), _stream(stream)),
           "fused_gemm_reduce_noalloc")


def fused_gemm_reduce_noalloc_status():
    """(code, detail) of the last fused_gemm_reduce_noalloc call on the current
    device; call after its work has completed (code 0: every wait finished)."""
    d = ctypes.c_int(0)
    code = int(_lib.fused_gemm_reduce_noalloc_status(ctypes.byref(d)))
    return code, int(d.value)
