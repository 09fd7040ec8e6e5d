"""The FMA-polynomial exp2 the kernel can use in place of the hardware unit.

Pinned against exp2 itself: the fitted coefficients in csrc/exp2_poly.h must
reproduce from the committed Remez script, meet the stated relative-error
bound on the reduced range, and -- with the kernel's float32 range reduction
and exponent-field scaling emulated here -- stay within that bound over the
whole range the softmax uses (x <= 8, the lazy-rescale threshold) without
ever wrapping the exponent field for very negative x.
"""
import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "attention_attn_fwd_04_gb300", "csrc")


def coeffs():
    text = open(os.path.join(CSRC, "exp2_poly.h")).read()
    c = [float.fromhex(re.search(r"ATTN_EXP2_POLY_C%d (\S+)f" % i, text).group(1)) for i in range(4)]
    err = float(re.search(r"ATTN_EXP2_POLY_MAX_REL_ERR (\S+)", text).group(1))
    return c, err


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def fma32(a, b, c):
    # one rounding of the exact a*b + c (float64 holds the float32 product exactly)
    return f32(a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64))


def kernel_exp2(x):
    """float32 emulation of ptx::exp2_poly."""
    c = [np.float32(v) for v in coeffs()[0]]
    x_in = f32(x)
    x = np.maximum(x_in, np.float32(-126.0))
    magic = np.float32(12582912.0)
    y = f32(x.astype(np.float64) + magic)
    f = f32(x.astype(np.float64) - f32(y.astype(np.float64) - magic))
    r = fma32(np.full_like(f, c[3]), f, np.full_like(f, c[2]))
    r = fma32(r, f, np.full_like(f, c[1]))
    r = fma32(r, f, np.full_like(f, c[0]))
    bits = r.view(np.int32).astype(np.int64) + (y.view(np.int32).astype(np.int64) << 23)
    e = (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    return np.where(x_in >= np.float32(-126.0), e, np.float32(0.0)).astype(np.float32)


def test_coefficients_reproduce_from_the_fit():
    spec = importlib.util.spec_from_file_location("gen", os.path.join(CSRC, "gen_exp2_poly.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    c = [float(np.float32(v)) for v in gen.remez()]
    assert c == coeffs()[0]


def test_reduced_range_error_bound():
    c, err = coeffs()
    x = np.linspace(-0.5, 0.5, 400001)
    p = np.polyval(np.array(c)[::-1], x)
    rel = np.abs(p - np.exp2(x)) / np.exp2(x)
    assert rel.max() <= 1.5e-4
    assert abs(rel.max() - err) <= 1e-3 * err + 1e-9
    # equal ripple: the error reaches its maximum at both interval ends
    assert rel[0] > 0.9 * rel.max() and rel[-1] > 0.9 * rel.max()


def test_full_range_with_float32_reduction():
    x = np.concatenate([np.linspace(-125.0, 8.0, 2000001), np.arange(-125, 9, dtype=np.float64),
                        np.arange(-125, 9) + 0.5])
    y = kernel_exp2(x).astype(np.float64)
    ref = np.exp2(f32(x).astype(np.float64))
    rel = np.abs(y - ref) / ref
    assert rel.max() <= 2e-4, rel.max()


def test_masked_and_very_negative_inputs_give_exactly_zero():
    # a hidden key (x = -inf) must add nothing to the row sum or to P V
    x = np.array([-126.7, -127.0, -300.0, -1e30, -np.inf], dtype=np.float32)
    assert np.all(kernel_exp2(x) == 0.0)
    # the smallest input still reduced: 2^-126, the smallest normal float32
    y = kernel_exp2(np.array([-126.0], dtype=np.float32))[0]
    assert abs(float(y) / 2.0 ** -126 - 1.0) <= 2e-4
