"""The C-ABI library loads and exports every entry point include/gemmar.h
declares; the host-only shape check answers without a GPU (CPU only: no
compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemmar.h")
LIB = os.path.join(ROOT, "block_scaled_fp8_gemm_gb300", "libgemmar.so")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:int|int64_t|void)\s+\**\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("gemmar_create", "gemmar_destroy", "gemmar_status", "gemm_blockscale_fp8", "gemm_mxfp8",
                     "band_reduce", "rowquant_e4m3", "rowdequant_e4m3", "fused_gemm_reduce"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_binding_covers_every_declared_symbol(lib):
    import block_scaled_fp8_gemm_gb300 as g
    assert sorted(g.EXPORTED) == declared_functions()
    for n in declared_functions():
        assert callable(getattr(g, n))


def test_shape_rules_host_only(lib):
    sup = lib.gemmar_supports
    sup.restype = ctypes.c_int
    sup.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    OK, ARG, SHAPE = 0, 1, 2
    assert sup(8, 16384, 7168, 2048, 8, 0) == OK        # the headline shape
    assert sup(4, 16384, 7168, 2048, 4, 1) == OK        # the mxfp8 shape
    assert sup(2, 256, 512, 256, 2, 0) == OK            # the tiny shape
    assert sup(8, 604, 7168, 2048, 8, 0) == SHAPE       # M not a multiple of the band count
    assert sup(8, 600, 7168, 2048, 8, 0) == OK          # ragged bands: 75 rows each
    assert sup(1, 200, 384, 256, 1, 0) == OK            # ragged M (one band)
    assert sup(1, 128, 7200, 2048, 1, 0) == SHAPE       # N off the 128 grid
    assert sup(1, 128, 448, 2048, 1, 0) == SHAPE        # blockscale N needs the 128 grid
    assert sup(1, 128, 448, 2048, 1, 1) == OK           # mx N may use the 224 tile
    assert sup(1, 128, 7168, 2000, 1, 0) == SHAPE       # K off the 128 grid
    assert sup(9, 128, 256, 128, 1, 0) == ARG           # more slices than the ABI takes
    assert sup(2, 128, 256, 128, 0, 0) == ARG
    assert sup(2, 128, 256, 128, 2, 7) == ARG           # unknown scale kind
    # empty inputs: zero rows, columns, K or slices are argument errors (nothing to launch)
    for empty in [(8, 0, 7168, 2048, 8, 0), (4, 0, 7168, 2048, 4, 1), (1, 128, 0, 2048, 1, 0),
                  (1, 128, 7168, 0, 1, 0), (0, 128, 256, 128, 1, 0)]:
        assert sup(*empty) == ARG, empty


def declared_constants():
    text = open(HEADER).read()
    consts = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", re.sub(r"/\*.*?\*/", "", text, flags=re.S), flags=re.S):
        for name, value in re.findall(r"(GEMMAR_[A-Z0-9_]+)\s*=\s*(\d+)", body):
            consts[name] = int(value)
    for name, expr in re.findall(r"^#define\s+(GEMMAR_[A-Z0-9_]+)\s+([^/\n]+)", text, flags=re.M):
        expr = expr.strip()
        m = re.fullmatch(r"\(\s*1u?\s*<<\s*(\d+)\s*\)", expr)
        if m:
            consts[name] = 1 << int(m.group(1))
            continue
        expr = expr.replace("u", "") if re.fullmatch(r"[\d\s\*\(\)u]+", expr) else expr
        try:
            consts[name] = int(eval(expr, {"__builtins__": {}}))
        except Exception:
            pass
    return consts


def test_binding_constants_match_the_header(lib):
    import block_scaled_fp8_gemm_gb300 as g
    consts = declared_constants()
    for required in ("GEMMAR_FP8_WIRE", "GEMMAR_FUSE_SLICES", "GEMMAR_FUSE_ONCHIP", "GEMMAR_CTA_PAIR",
                     "GEMMAR_SCALE_BLOCK128", "GEMMAR_SCALE_MX32"):
        assert required in consts, required
    for name, value in consts.items():
        if hasattr(g, name):
            assert getattr(g, name) == value, (name, getattr(g, name), value)
    # every flag bit is distinct
    flag_names = ("GEMMAR_FP8_WIRE", "GEMMAR_DEBUG_CANARY", "GEMMAR_FAULT_SKIP_BAND", "GEMMAR_NO_SELF_TEST",
                  "GEMMAR_FUSE_SLICES", "GEMMAR_CTA_PAIR", "GEMMAR_FUSE_ONCHIP", "GEMMAR_SERIAL_REDUCE",
                  "GEMMAR_FUSE_QUANTIZE")
    flags = [consts[n] for n in flag_names]
    assert len(flags) == len(set(flags)) == len(flag_names)
    assert all(f & (f - 1) == 0 for f in flags)   # one bit each


def test_host_side_argument_errors(lib):
    """Entry points that take a context refuse a null one before touching the GPU."""
    ARG = 1
    st = lib.gemmar_overlap_stats
    st.restype = ctypes.c_int
    st.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
    a, b = ctypes.c_int64(7), ctypes.c_int64(7)
    assert st(None, ctypes.byref(a), ctypes.byref(b)) == ARG
    ps = lib.gemmar_phase_times
    ps.restype = ctypes.c_int
    ps.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]
    assert ps(None, None, None) == ARG
