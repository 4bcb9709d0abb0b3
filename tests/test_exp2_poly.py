"""The FMA-pipe 2^x of the attention kernels (common.cuh, exp2_poly2), on the
CPU: its coefficients are the output of the committed fit script, and its
error bounds hold -- the polynomial's maximum relative error on [-1/2, 1/2]
in float64, and the whole float32 evaluation (Cody-Waite split, Horner with
fused multiply-adds, exponent add) against numpy's float64 2^x over
[-125, 128].  The GPU test in test_gpu_diagnostics.py checks the kernel's
own outputs against the same bound.
"""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "partial_attention_saliency_b300", "csrc")
sys.path.insert(0, CSRC)

import fit_exp2_poly  # noqa: E402

BOUND = 2.7e-6


def header_coefficients():
    """The float32 coefficients in exp2_poly2, highest degree first."""
    src = open(os.path.join(CSRC, "common.cuh")).read()
    body = src[src.index("exp2_poly2(float2 x)"):]
    body = body[:body.index("return")]
    lits = re.findall(r"make_float2\((0x[0-9a-fA-F.]+p-?\d+)f,", body)
    return [np.float32(float.fromhex(v)) for v in lits]


def test_coefficients_are_the_fit_scripts():
    c32, err = fit_exp2_poly.fit()
    assert [float(v) for v in header_coefficients()] == [float(v) for v in c32[::-1]]
    assert err <= 2.65e-6


def emulate(x):
    """exp2_poly2 step by step in float32 (a fused multiply-add rounds once:
    the product of two float32 values is exact in float64)."""
    c = header_coefficients()
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    sh = np.float32(12582912.0)
    t = x + sh
    n = t - sh
    f = x - n
    p = np.full_like(f, c[0])
    for ck in c[1:]:
        p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(ck)).astype(np.float32)
    bits = (p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23))
    return (bits & 0xffffffff).astype(np.uint32).view(np.float32)


def test_float32_evaluation_within_bound():
    x = np.linspace(-125.0, 128.0, 2_000_001).astype(np.float32)
    y = emulate(x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() <= BOUND, (rel.max(), x[rel.argmax()])
    # integers are exact up to the polynomial's value at 0
    k = np.arange(-125, 129).astype(np.float32)
    assert np.all(np.abs(emulate(k).astype(np.float64) / np.exp2(k.astype(np.float64)) - 1) <= BOUND)
