"""CPU oracle for the block-scaled fp8 wo_b path (plain C in ``oracle.c``, fp64).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()``, and
``bench.py``'s CPU-baseline leg (which also checks the GPU result on its sample)
and its ``--impl reference`` arm are the only callers.  The CUDA library never
imports, links or executes anything here, and this module imports nothing
from the CUDA package.

Every function cites the page passage it follows (see ``oracle.c``).  All are
pinned by ``tests/test_oracle_*.py`` against values the pages print, closed
forms, library routines or exact rational brute force.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build as _build, LIB_PATH

_lib = None


def lib() -> ctypes.CDLL:
    """Load (building on first use) the oracle shared library."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(
            os.path.join(os.path.dirname(__file__), "oracle.c")
        ):
            _build()
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_decode_table.argtypes = [P]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode_array.argtypes = [P, i64, P]
        L.orc_bf16_rn.restype = ctypes.c_uint16
        L.orc_bf16_rn.argtypes = [ctypes.c_double]
        L.orc_bf16_rn_array.argtypes = [P, i64, P]
        L.orc_quant_block.argtypes = [P, i64, i64, i64, i64, P, P]
        L.orc_ue8m0_byte.restype = ctypes.c_uint8
        L.orc_ue8m0_byte.argtypes = [ctypes.c_float]
        L.orc_quant_mx.argtypes = [P, i64, i64, P, P]
        L.orc_gemm_blockscale_acc.argtypes = [P, P, P, P, i64, i64, i64, P, i64, P]
        L.orc_gemm_mx_acc.argtypes = [P, P, P, P, i64, i64, i64, P, i64, P]
        L.orc_gemm_reduce.argtypes = [ctypes.c_int, P, P, P, P, ctypes.c_int,
                                      i64, i64, i64, P, i64, P, P]
        L.orc_reduce_f32_ordered.argtypes = [ctypes.c_int, P, i64, i64, P]
        L.orc_rowquant.argtypes = [P, i64, i64, P, P]
        L.orc_rowdequant.argtypes = [P, P, i64, i64, P]
        L.orc_bf16_to_f32.argtypes = [P, i64, P]
        L.orc_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    return int(lib().orc_num_threads())


# --- e4m3 / bf16 primitives ------------------------------------------------

def e4m3_decode_table() -> np.ndarray:
    out = np.empty(256, dtype=np.float64)
    lib().orc_e4m3_decode_table(_p(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def bf16_rn(x) -> np.ndarray:
    """Round fp64 values once to bf16 (nearest-even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_bf16_rn_array(_p(x), x.size, _p(out))
    return out


def bf16_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    lib().orc_bf16_to_f32(_p(b), b.size, _p(out))
    return out


def ue8m0_byte(r: float) -> int:
    return int(lib().orc_ue8m0_byte(ctypes.c_float(r)))


# --- quantisers ------------------------------------------------------------

def quant_block(x: np.ndarray, gr: int, gc: int):
    """Quantise a 2-D fp32 matrix in gr x gc groups -> (codes uint8, scales fp32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    codes = np.empty((R, C), dtype=np.uint8)
    scales = np.empty(((R + gr - 1) // gr, (C + gc - 1) // gc), dtype=np.float32)
    lib().orc_quant_block(_p(x), R, C, gr, gc, _p(codes), _p(scales))
    return codes, scales


def quant_act_1x128(x):
    return quant_block(x, 1, 128)


def quant_weight_128x128(x):
    return quant_block(x, 128, 128)


def quant_mx(x: np.ndarray):
    """mxfp8 quantiser: 1x32 groups, ue8m0 bytes -> (codes uint8, bytes uint8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    codes = np.empty((R, C), dtype=np.uint8)
    sb = np.empty((R, (C + 31) // 32), dtype=np.uint8)
    lib().orc_quant_mx(_p(x), R, C, _p(codes), _p(sb))
    return codes, sb


def quant_ptpc(x: np.ndarray):
    """ptpc quantiser: one fp32 scale per row over the whole row (per token for
    A [M,K], per output channel for B [N,K]) -> (codes uint8, scales fp32 [R])."""
    codes, scales = quant_block(x, 1, np.asarray(x).shape[1])
    return codes, np.ascontiguousarray(scales[:, 0])


# --- GEMM + reduction --------------------------------------------------------

def gemm_reduce(A, sa, B, sb, scale_kind: int = 0, rows=None, want_ref: bool = True):
    """fp64 P-way sum of per-slice scaled GEMMs for the listed rows.

    A, sa, B, sb are lists of P numpy arrays (A_p [M,K] uint8, B_p [N,K] uint8;
    sa/sb fp32 block scales for scale_kind 0, ue8m0 bytes for scale_kind 1,
    fp32 per-row scales sa [M] and sb [N] for scale_kind 2, ptpc).
    Returns (ref fp64 [nrows,N] or None, out bf16 bits uint16 [nrows,N]).
    """
    P = len(A)
    M, K = A[0].shape
    N = B[0].shape[0]
    A = [np.ascontiguousarray(a) for a in A]
    B = [np.ascontiguousarray(b) for b in B]
    sa = [np.ascontiguousarray(s) for s in sa]
    sb = [np.ascontiguousarray(s) for s in sb]
    arrA = (ctypes.c_void_p * P)(*[a.ctypes.data for a in A])
    arrB = (ctypes.c_void_p * P)(*[b.ctypes.data for b in B])
    arrSA = (ctypes.c_void_p * P)(*[s.ctypes.data for s in sa])
    arrSB = (ctypes.c_void_p * P)(*[s.ctypes.data for s in sb])
    if rows is None:
        nrows = M
        rows_p = ctypes.c_void_p(0)
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
        rows_p = _p(rows_arr)
    ref = np.empty((nrows, N), dtype=np.float64)
    out = np.empty((nrows, N), dtype=np.uint16)
    lib().orc_gemm_reduce(P, arrA, arrSA, arrB, arrSB, scale_kind, M, N, K, rows_p, nrows,
                          _p(ref), _p(out))
    return (ref if want_ref else None), out


def reduce_f32_ordered(W: np.ndarray):
    """W [P, rows, N] fp32 -> bf16 bits of the fp32 sum taken in order p = 0..P-1."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    P, R, N = W.shape
    out = np.empty((R, N), dtype=np.uint16)
    lib().orc_reduce_f32_ordered(P, _p(W), R, N, _p(out))
    return out


# --- fp8 wire codec ------------------------------------------------------------

def rowquant(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, N = x.shape
    q = np.empty((M, N), dtype=np.uint8)
    s = np.empty((M,), dtype=np.float32)
    lib().orc_rowquant(_p(x), M, N, _p(q), _p(s))
    return q, s


def rowdequant(q: np.ndarray, s: np.ndarray):
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    M, N = q.shape
    y = np.empty((M, N), dtype=np.uint16)
    lib().orc_rowdequant(_p(q), _p(s), M, N, _p(y))
    return y
