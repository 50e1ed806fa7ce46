"""Shared helpers for the parity tests: seeded operands (drawn by `synthetic`,
quantised by the oracle on the host, so both sides consume identical codes and
scales) and the tolerance checks written in the tests."""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
import synthetic

# the bf16 GEMM+reduce tolerance against the fp64 oracle
REL_L2_MAX = 4e-3
ELEM_REL = 1e-2
ELEM_ABS = 1e-3

# The pages' measured relL2 of the fused output against an fp32 host reference
# (MORI GEMM + All-Reduce Benchmark, "What fp8 costs, numerically"): 2.35e-3
# with bf16 partials on the wire.  fp32 partials must land below it.
with open(os.path.join(os.path.dirname(__file__), "golden", "mori_numerics_levels.json")) as _f:
    _LEVELS = json.load(_f)
PAGES_BF16_WIRE_REL_L2 = float(_LEVELS["rel_l2_bf16_wire"])
PAGES_FP8_WIRE_REL_L2 = float(_LEVELS["rel_l2_fp8_wire"])


def blockscale_operands(P, M, N, K, seed=0):
    A, sa, B, sb = [], [], [], []
    for p in range(P):
        a, s = oracle.quant_act_1x128(synthetic.normal(seed, synthetic.TID_A, p, (M, K)))
        b, t = oracle.quant_weight_128x128(synthetic.normal(seed, synthetic.TID_B, p, (N, K), sigma=0.02))
        A.append(a); sa.append(s); B.append(b); sb.append(t)
    return A, sa, B, sb


def mx_operands(P, M, N, K, seed=0):
    A, sa, B, sb = [], [], [], []
    for p in range(P):
        a, s = oracle.quant_mx(synthetic.normal(seed, synthetic.TID_A, p, (M, K)))
        b, t = oracle.quant_mx(synthetic.normal(seed, synthetic.TID_B, p, (N, K), sigma=0.02))
        A.append(a); sa.append(s); B.append(b); sb.append(t)
    return A, sa, B, sb


def ptpc_operands(P, M, N, K, seed=0):
    """Per-token A and per-channel B scales (one fp32 scale per row of each)."""
    A, sa, B, sb = [], [], [], []
    for p in range(P):
        a, s = oracle.quant_ptpc(synthetic.normal(seed, synthetic.TID_A, p, (M, K)))
        b, t = oracle.quant_ptpc(synthetic.normal(seed, synthetic.TID_B, p, (N, K), sigma=0.02))
        A.append(a); sa.append(s); B.append(b); sb.append(t)
    return A, sa, B, sb


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def check_bf16_output(got, ref, what=""):
    """relL2 <= 4e-3 and |err| <= 1e-2 |ref| + 1e-3 elementwise (fp64 reference)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs (unwritten tiles?)"
    rl = rel_l2(got, ref)
    err = np.abs(got - ref)
    bad = err > ELEM_REL * np.abs(ref) + ELEM_ABS
    assert rl <= REL_L2_MAX, f"{what}: relL2 {rl:.3e} > {REL_L2_MAX}"
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of bound, worst {err[bad].max():.3e}"
    return rl


def check_f32_output(got, ref, what=""):
    """An fp32 single-slice GEMM against fp64: fp32 accumulation and promotion
    cost a few fp32 roundings of the magnitudes involved."""
    got = np.asarray(got, np.float64)
    scale = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), what
    assert rel_l2(got, ref) <= 2e-6, (what, rel_l2(got, ref))
    assert np.all(err <= 1e-5 * np.abs(ref) + 2e-5 * scale), (what, err.max())
