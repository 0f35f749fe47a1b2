"""CPU pin of the FMA-pipe exponential's fit: the same range reduction and
polynomial, emulated step by step in float32, against 2^x in double precision.

The kernel's function (Cody-Waite reduction x = n + f, n = rint(x) via adding
1.5 * 2^23, a degree-5 polynomial for 2^f on [-1/2, 1/2], exponent add) is
restated here from its mathematics; the coefficients are read from the CUDA
header so that a changed coefficient fails here before it reaches a GPU.
"""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(__file__), "..", "top_block_sparse_pooled_b300", "csrc", "sa_exp2.cuh")


def _coefficients():
    body = open(HDR).read()
    lead = re.search(r"float p = ([0-9.eE+-]+)f;", body).group(1)
    rest = re.findall(r"p = fmaf\(p, f, ([0-9.eE+-]+)f\);", body)
    return [np.float32(v) for v in [lead] + rest]


def _exp2_poly32(x):
    f32 = np.float32
    c = _coefficients()
    t = (x + f32(12582912.0)).astype(np.float32)
    f = (x - (t - f32(12582912.0)).astype(np.float32)).astype(np.float32)
    p = np.full_like(f, c[0])
    for ci in c[1:]:  # fma: exact product, one rounding (float64 holds the product exactly)
        p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(ci)).astype(np.float32)
    e = (t.view(np.int32).astype(np.int64) << 23) & 0xFFFFFFFF
    y = ((p.view(np.int32).astype(np.int64) + e) & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    return np.where(x < -126.0, np.float32(0.0), y)


def test_fit_is_degree_five_and_near_taylor():
    c = _coefficients()
    assert len(c) == 6
    # the leading terms of 2^f = sum (ln 2)^k f^k / k!, highest degree first
    taylor = [np.log(2) ** k / np.prod(range(1, k + 1)) for k in range(5, -1, -1)]
    assert np.allclose(c, taylor, rtol=0.02)


def test_reduced_range_error():
    f = np.linspace(-0.5, 0.5, 200_001)
    c = [float(v) for v in _coefficients()]
    p = np.polyval(c, f)
    assert np.max(np.abs(p / np.exp2(f) - 1.0)) < 1.1e-7
    assert c[-1] == 1.0  # 2^0 exactly


def test_float32_emulation_error():
    rng = np.random.default_rng(3)
    x = np.concatenate([np.linspace(-126, 0, 400_001), rng.uniform(-126, 0, 400_000),
                        np.arange(-126, 1), np.arange(-126, 0) + 0.5]).astype(np.float32)
    y = _exp2_poly32(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(y - ref) / ref) < 2.5e-7
    assert np.all(_exp2_poly32(np.array([-126.5, -200.0, -np.inf], dtype=np.float32)) == 0.0)
