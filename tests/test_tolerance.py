"""CPU checks of the parity criterion's helpers (tests/tolerance.py): the
bf16 rounding and spacing against torch's own float32 -> bf16 conversion,
and the criterion's pass / excuse / fail decisions on planted errors."""
import numpy as np
import pytest
import torch

import tolerance


def test_bf16_rne_matches_torch_conversion():
    g = torch.Generator().manual_seed(5)
    x = torch.cat([torch.randn(100000, generator=g) * s for s in (1e-3, 1.0, 7.0, 1e4)])
    # float32 inputs are exact in float64; torch rounds float32 to bf16 to
    # nearest, ties to even
    want = x.to(torch.bfloat16).double().numpy()
    got = tolerance.bf16_rne(x.double().numpy())
    np.testing.assert_array_equal(got, want)
    # ties go to the even neighbour: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert tolerance.bf16_rne(1.0 + 2.0 ** -8) == 1.0
    assert tolerance.bf16_rne(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6


def test_bf16_ulp_is_the_spacing():
    for y, u in ((1.0, 2.0 ** -7), (1.99, 2.0 ** -7), (2.0, 2.0 ** -6), (4.5, 2.0 ** -5),
                 (-6.0, 2.0 ** -5), (0.25, 2.0 ** -9), (0.0, 0.0)):
        assert tolerance.bf16_ulp(y) == u, y
    # the next bf16 value above y is y + ulp
    g = torch.Generator().manual_seed(6)
    y = torch.randn(1000, generator=g).abs().to(torch.bfloat16)
    bits = y.view(torch.int16).numpy().astype(np.int64) + 1
    above = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(above - y.double().numpy(), tolerance.bf16_ulp(y.double().numpy()))


def rows(n=64, D=8, seed=0):
    g = np.random.default_rng(seed)
    ro = 0.3 * g.standard_normal((n, D))  # attention outputs average many values
    rl = g.standard_normal(n)
    return ro, rl


def test_criterion_passes_rounded_oracle():
    ro, rl = rows()
    tolerance.check(tolerance.bf16_rne(ro), rl + 1e-4, ro, rl)


def test_criterion_fails_error_above_tolerance():
    ro, rl = rows()
    go = tolerance.bf16_rne(ro)
    go[3, 2] += 0.02  # |O| < 2 here: 0.02 is more than one bf16 spacing
    with pytest.raises(AssertionError):
        tolerance.check(go, rl, ro, rl)


def test_criterion_excuses_one_ulp_at_large_magnitude_only():
    ro, rl = rows()
    ro[5, 1] = 5.0 + 0.011  # bf16 spacing at 5 is 2^-5 = 0.03125
    go = tolerance.bf16_rne(ro)
    go[5, 1] = 5.0 + 2.0 ** -5  # 0.0202 from O_ref, one spacing from bf16(O_ref) = 5
    msg = tolerance.check(go, rl, ro, rl)
    assert "1 of them within 1 bf16 ulp" in msg
    go[5, 1] = 5.0 + 2 * 2.0 ** -5  # two spacings away: fails
    with pytest.raises(AssertionError):
        tolerance.check(go, rl, ro, rl)


def test_criterion_bounds_the_excused_count():
    ro, rl = rows(n=64, D=8)
    ro[:, 0] = 5.011
    go = tolerance.bf16_rne(ro)
    go[:, 0] = 5.0 + 2.0 ** -5  # 64 excusable elements, above max(8, 1e-4 n)
    with pytest.raises(AssertionError):
        tolerance.check(go, rl, ro, rl)


def test_criterion_checks_lse_mean_and_empty_rows():
    ro, rl = rows()
    go = tolerance.bf16_rne(ro)
    with pytest.raises(AssertionError):
        tolerance.check(go, rl + 2e-3, ro, rl)
    with pytest.raises(AssertionError):
        tolerance.check(go + 2e-3, rl, ro, rl)  # mean |dO| above 1e-3
    rl2 = rl.copy()
    rl2[7] = -np.inf
    ro2 = ro.copy()
    ro2[7] = 0
    go2 = tolerance.bf16_rne(ro2)
    tolerance.check(go2, rl2, ro2, rl2)
    with pytest.raises(AssertionError):
        tolerance.check(go2, rl, ro2, rl2)  # GPU LSE finite where the oracle's is -inf
