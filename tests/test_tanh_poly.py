"""The soft cap's tanh polynomial (csrc/tanh_poly.h), pinned against tanh
itself: the coefficients reproduce from the fit script, the float32
evaluation the kernel performs (coefficients pre-scaled on the host for the
raw score or for the biased score) matches cap * log2(e) * tanh(x / cap) over
the whole range where the kernel uses it, and a masked score (NaN on a
partial tile) gives an exponent of -inf, so its exponential is exactly 0."""
import importlib.util
import os
import re

import numpy as np
import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "attention_attn_fwd_04_gb300", "csrc")
L2E = 1.4426950408889634
f32 = np.float32


def header():
    text = open(os.path.join(CSRC, "tanh_poly.h")).read()
    r = [float.fromhex(re.search(r"ATTN_TANH_POLY_R%d (\S+)" % i, text).group(1))
         for i in range(3)]
    assert "ATTN_TANH_POLY_R3" not in text
    u0 = float(re.search(r"ATTN_TANH_POLY_U0 (\S+)", text).group(1))
    err = float(re.search(r"ATTN_TANH_POLY_MAX_ABS_ERR (\S+)", text).group(1))
    return r, u0, err


def host_coefficients(scale, cap, biased):
    """What the launcher computes: tq_i = cap log2e R_i kk^(2i+1), the range
    limit U0 / kk and the fallback factor, with u = kk v."""
    r, u0, _ = header()
    kk = 1.0 / (2.0 * L2E) if biased else scale / cap
    C = cap * L2E
    tq = [f32(C * r[i] * kk ** (2 * i + 1)) for i in range(3)]
    return tq, f32(u0 / kk), kk


def kernel_eval(v, tq):
    """float32 emulation of the kernel: w = v v; Horner with fma; t = v q."""
    v = np.asarray(v, dtype=f32)
    with np.errstate(invalid="ignore", over="ignore"):
        w = (v.astype(np.float64) * v).astype(f32)
        q = (w.astype(np.float64) * tq[2] + np.float64(tq[1])).astype(f32)
        q = (q.astype(np.float64) * w + np.float64(tq[0])).astype(f32)
        return (v.astype(np.float64) * q).astype(f32)


def test_coefficients_reproduce_from_the_fit():
    spec = importlib.util.spec_from_file_location("gen", os.path.join(CSRC, "gen_tanh_poly.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    r, u0, err = header()
    assert [float(c) for c in gen.remez()] == r
    assert u0 == gen.U0
    assert abs(gen.max_abs_err_f32(gen.remez()) - err) <= 1e-3 * err


def test_relative_error_of_the_fit_on_the_range():
    r, u0, _ = header()
    u = np.linspace(-u0, u0, 400001)
    p = u * np.polyval(np.asarray(r)[::-1], u * u)
    rel = np.abs(p - np.tanh(u)) / np.maximum(np.abs(np.tanh(u)), 1e-300)
    assert rel[np.abs(u) > 1e-6].max() <= 7e-6


@pytest.mark.parametrize("scale,cap,biased", [(1 / np.sqrt(128), 30.0, False),
                                              (1 / np.sqrt(64), 5.0, False),
                                              (0.5, 50.0, False),
                                              (1 / np.sqrt(128), 30.0, True),
                                              (1 / np.sqrt(64), 2.0, True)])
def test_scaled_evaluation_matches_the_soft_cap(scale, cap, biased):
    tq, tlim, kk = host_coefficients(scale, cap, biased)
    v = np.linspace(-float(tlim), float(tlim), 200001).astype(f32)
    got = kernel_eval(v, tq).astype(np.float64)
    want = cap * L2E * np.tanh(kk * v.astype(np.float64))
    # the polynomial's 2.4e-6 in tanh times cap log2(e), plus float32
    # rounding: at cap 30 about 1e-4 of an exponent, far below the bf16
    # rounding of P (2^-9 relative)
    assert np.abs(got - want).max() <= 2.6e-6 * cap * L2E + 2e-7 * np.abs(want).max()


def test_masked_scores_give_minus_infinity():
    # a hidden score is NaN on a partial tile: the exponent argument
    # v Q(v^2) - m is NaN, and fmaxf(NaN, -inf) (IEEE maxNum, as the GPU's
    # max.f32) turns it into -inf, whose exponential is exactly 0
    for biased in (False, True):
        tq, _, _ = host_coefficients(1 / np.sqrt(128), 30.0, biased)
        t = kernel_eval(np.array([np.nan], dtype=f32), tq).astype(np.float64) - 3.0
        a = np.fmax(t, -np.inf)
        assert a[0] == -np.inf and np.exp2(a[0]) == 0.0
    # visible scores pass through unchanged
    tq, tlim, _ = host_coefficients(1 / np.sqrt(128), 30.0, False)
    v = np.linspace(-float(tlim), float(tlim), 1001).astype(f32)
    t = kernel_eval(v, tq)
    assert np.array_equal(np.fmax(t, f32(-np.inf)), t)
