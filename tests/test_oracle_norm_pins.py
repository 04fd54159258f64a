"""Pins for the oracle's deterministic gradient norm (CPU only).

The bins must reproduce, exactly, what the mathematics fixes independently of
them: the correctly rounded sum of the FP32 squares (``math.fsum``), closed
forms, the FP32 rounding of a square, subnormal and overflowing squares, and
invariance under any split of the elements across "ranks".  Planted mistakes
at the end must each fail at least one pin.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import norm_oracle as no


def _rng_vectors():
    rng = np.random.default_rng(5)
    yield (1e-3 * rng.standard_normal(5000)).astype(np.float32)
    # exponents spread over the whole finite FP32 square range
    yield (rng.choice([-1, 1], 3000) * 2.0 ** rng.uniform(-80, 60, 3000)).astype(np.float32)
    yield rng.standard_normal(777).astype(np.float32)


def pin_fsum(impl):
    """Sum of squares == math.fsum of the FP32 squares (exactly rounded sum)."""
    for x in _rng_vectors():
        q = (x * x).astype(np.float64)
        want = math.fsum(q.tolist())
        s, n = impl(x, "f32")
        assert s == want, (s, want)
        assert n == math.sqrt(want)


def pin_closed_forms(impl):
    assert impl(np.array([3.0, 4.0], np.float32), "f32") == (25.0, 5.0)
    assert impl(np.ones(10, np.float32), "f32") == (10.0, math.sqrt(10.0))
    assert impl(np.zeros(0, np.float32), "f32") == (0.0, 0.0)
    assert impl(np.array([-2.0, 0.0, 0.5], np.float32), "f32") == (4.25, math.sqrt(4.25))


def pin_fp32_square_rounding(impl):
    """(1 + 2^-23)^2 = 1 + 2^-22 + 2^-46 rounds to 1 + 2^-22 in FP32."""
    assert impl(np.array([1.0 + 2.0 ** -23], np.float32), "f32")[0] == 1.0 + 2.0 ** -22


def pin_subnormal_squares(impl):
    """2^-70 squares to the subnormal 2^-140; 2^-75 squares to 2^-150, a tie
    that rounds to 0; 1.5 * 2^-75 squares to 1.125 * 2^-149, which rounds to
    the smallest subnormal."""
    assert impl(np.array([2.0 ** -70], np.float32), "f32")[0] == 2.0 ** -140
    assert impl(np.array([2.0 ** -75], np.float32), "f32")[0] == 0.0
    assert impl(np.array([1.5 * 2.0 ** -75], np.float32), "f32")[0] == 2.0 ** -149
    assert impl(np.array([2.0 ** -70, 3.0], np.float32), "f32")[0] == 9.0 + 2.0 ** -140


def pin_specials(impl):
    f = lambda v: impl(np.array(v, np.float32), "f32")
    assert all(math.isnan(r) for r in f([1.0, np.nan]))
    assert f([np.inf, 1.0]) == (math.inf, math.inf)
    assert all(math.isnan(r) for r in f([np.inf, np.nan]))
    assert f([2.0 ** 64]) == (math.inf, math.inf)          # the FP32 square overflows
    s, _ = f([1.8e19, 1.8e19])                             # finite squares, sum above FP32 max
    assert s == 2 * float(np.float32(np.float32(1.8e19) * np.float32(1.8e19)))


def pin_exact_not_naive(impl):
    """2^54 + 1 + 1 + 1: the exact sum 2^54 + 3 rounds to 2^54 + 4, while a
    left-to-right float64 sum stays at 2^54."""
    assert impl(np.array([2.0 ** 27, 1, 1, 1], np.float32), "f32")[0] == 2.0 ** 54 + 4


def pin_partition_invariance(impl_bins):
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(4000) * 2.0 ** rng.uniform(-30, 30, 4000)).astype(np.float32)
    whole = oracle.norm_finalize(impl_bins(x, "f32"))
    for parts in (2, 3, 8):
        cuts = np.sort(rng.choice(np.arange(1, len(x)), parts - 1, replace=False))
        b = sum(impl_bins(p, "f32").astype(object) for p in np.split(rng.permutation(x), cuts))
        assert oracle.norm_finalize(np.array(b, dtype=np.uint64)) == whole


def pin_half_inputs(impl):
    """BF16 bit patterns and FP16 values convert exactly."""
    bf = np.array([0x4040, 0x4080], np.uint16)                 # 3.0, 4.0
    assert impl(bf, "bf16") == (25.0, 5.0)
    assert impl(np.array([3.0, 4.0], np.float16), "f16") == (25.0, 5.0)
    assert impl(np.array([2.0 ** -24], np.float16), "f16")[0] == 2.0 ** -48   # FP16 subnormal


NORM_PINS = [pin_fsum, pin_closed_forms, pin_fp32_square_rounding, pin_subnormal_squares,
             pin_specials, pin_exact_not_naive, pin_half_inputs]


@pytest.mark.parametrize("pin", NORM_PINS, ids=lambda f: f.__name__)
def test_norm_pin(pin):
    pin(oracle.grad_norm)


def test_norm_partition_invariance():
    pin_partition_invariance(oracle.sqnorm_bins)


def test_bins_layout():
    b = oracle.sqnorm_bins(np.array([1.0, 1.0, 0.5, np.nan, np.inf], np.float32))
    assert b.dtype == np.uint64 and len(b) == oracle.NORM_BINS
    assert b[127] == 2 * (1 << 23) and b[125] == 1 << 23          # 1.0 = 2^23 * 2^(127-150)
    assert b[oracle.NAN_BIN] == 1 and b[oracle.INF_BIN] == 1
    assert oracle.bins_exact(b) == (2 << 149) + (1 << 147)


# ------------------------------------------------------ planted mistakes

def _sum_with(x, dtype, *, implicit=True, bias=150, sub_bin=1):
    """The bins' exact sum with one step of the split changed (exact integer
    arithmetic in units of 2^-200, correctly rounded at the end)."""
    u = oracle.fp32_squares(x, dtype).view(np.uint32)
    total = 0
    for w in u.tolist():
        Ei, fi = (w >> 23) & 0xFF, w & 0x7FFFFF
        if Ei == 255:
            return math.nan if fi else math.inf
        M = (fi | (1 << 23)) if (Ei > 0 and implicit) else fi
        e = Ei if Ei > 0 else sub_bin
        total += M << (e - bias + 200)
    return total / (1 << 200)


def _mut_no_implicit_bit(x, dtype):
    s = _sum_with(x, dtype, implicit=False)
    return s, math.sqrt(s) if s == s else s


def _mut_bias_off_by_one(x, dtype):
    s = _sum_with(x, dtype, bias=149)
    return s, math.sqrt(s) if s == s else s


def _mut_subnormal_bin0(x, dtype):
    """Mistake: subnormal squares get the weight of a bin 0 (2^-150 per unit)."""
    s = _sum_with(x, dtype, sub_bin=0)
    return s, math.sqrt(s) if s == s else s


def _mut_f64_squares(x, dtype):
    q = no.to_f32(x, dtype).astype(np.float64) ** 2
    s = math.fsum(q.tolist())
    return s, math.sqrt(s)


def _mut_naive_float_sum(x, dtype):
    s = 0.0
    for v in oracle.fp32_squares(x, dtype).astype(np.float64).tolist():
        s += v
    return s, math.sqrt(s) if s == s else s


def _mut_nan_as_inf(x, dtype):
    s, n = oracle.grad_norm(x, dtype)
    return (math.inf, math.inf) if s != s else (s, n)


@pytest.mark.parametrize("mutant", [_mut_no_implicit_bit, _mut_bias_off_by_one, _mut_subnormal_bin0,
                                    _mut_f64_squares, _mut_naive_float_sum, _mut_nan_as_inf],
                         ids=lambda f: f.__name__)
def test_planted_norm_mistake_is_caught(mutant):
    failed = []
    for pin in NORM_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, OverflowError):
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"


def test_norm_equals_fsum_on_random_float32_arrays():
    """Property: for any FP32 array (any exponents, subnormals, zeros), the
    oracle's sum of squares is math.fsum of the FP32 squares."""
    hypothesis = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hypothesis.settings(max_examples=200, deadline=None)
    @hypothesis.given(st.lists(st.floats(width=32, allow_nan=False, allow_infinity=False),
                               min_size=0, max_size=64))
    def check(vals):
        x = np.array(vals, dtype=np.float32)
        with np.errstate(over="ignore", under="ignore"):
            q = (x * x).astype(np.float64)
        if not np.all(np.isfinite(q)):
            assert oracle.grad_norm(x, "f32") == (math.inf, math.inf)
            return
        want = math.fsum(q.tolist())
        assert oracle.grad_norm(x, "f32") == (want, math.sqrt(want))

    check()
