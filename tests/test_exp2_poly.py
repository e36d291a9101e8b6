"""The FMA-pipe 2^x of zl_exp2.cuh, emulated step by step on the CPU: float32 rounding of
every operation (the fused multiply-adds rounded once), the round-to-integer by adding
1.5 * 2^23, and the exponent insertion by an integer multiply-add modulo 2^32.  The
coefficients are read from the header itself.  Checked against float64 exp2: the worst
relative error stays within the bound the header states, over the whole clamped range and
for arguments above 0 (a lagging running maximum gives exponents up to +8)."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "coalesced_packed_attention_gb300", "csrc", "zl_exp2.cuh")


def coefficients(degree):
    txt = open(HDR).read()
    m = re.search(r"struct Exp2Poly<%d> \{\s*static constexpr float c\[%d\] = \{([^}]*)\}" % (degree, degree + 1), txt)
    return [np.float32(float.fromhex(v.strip().rstrip("f"))) for v in m.group(1).split(",")]


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def fma32(a, b, c):
    return f32(a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64))


def exp2_device(x, degree):
    c = coefficients(degree)
    x = np.maximum(f32(x), np.float32(-125.0))
    r = np.float32(12582912.0)
    t = f32(x.astype(np.float64) + r)
    j = f32(t.astype(np.float64) - r)
    f = f32(x.astype(np.float64) - j)
    p = np.full_like(f, c[degree])
    for k in range(degree - 1, -1, -1):
        p = fma32(p, f, np.full_like(f, c[k]))
    bits = (t.view(np.uint32).astype(np.uint64) * (1 << 23) + p.view(np.uint32).astype(np.uint64)) % (1 << 32)
    return bits.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("degree,bound", [(3, 7.5e-5), (4, 2.8e-6)])
def test_exp2_poly_relative_error(degree, bound):
    x = np.concatenate([np.linspace(-124.9, 8.5, 400001), np.linspace(-2, 2, 100001),
                        np.array([0.0, -0.5, 0.5, -1.0, -124.5, -125.0, 8.0], dtype=np.float64)])
    x = f32(x)
    got = exp2_device(x, degree).astype(np.float64)
    ref = np.exp2(np.maximum(x.astype(np.float64), -125.0))
    assert np.all(np.isfinite(got)) and np.all(got > 0)
    rel = np.abs(got / ref - 1.0)
    assert rel.max() <= bound, rel.max()


def test_exp2_poly_clamps_far_below():
    # arguments below -125 (never masked ones: callers use MUFU there) give 2^-125 * p(0)
    got = exp2_device(f32([-126.0, -1000.0, -3.0e38]), 4).astype(np.float64)
    assert np.allclose(got, 2.0 ** -125, rtol=1e-5)


def test_round_to_integer_trick_matches_rint():
    x = f32(np.linspace(-125.0, 9.0, 100003))
    t = f32(x.astype(np.float64) + 12582912.0)
    assert np.array_equal(f32(t.astype(np.float64) - 12582912.0), np.rint(x))
    inc = (t.view(np.uint32).astype(np.uint64) * (1 << 23)) % (1 << 32)
    assert np.array_equal(inc.astype(np.uint32).view(np.int32), (np.rint(x).astype(np.int64) << 23).astype(np.int32))
