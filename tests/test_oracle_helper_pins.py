"""Pins for the oracle's helper functions (CPU only).

Three helpers of the oracle serve the GPU tests directly:

* ``linear_logp_rows`` checks the fused LM-head kernel (row loop over
  ``linear_logp_row`` with per-row temperatures);
* ``row_logprobs_all`` draws every parity test's targets and scores the
  sampler's frequencies (the full and restricted logprob of every token);
* ``restr_for_support_size`` scores a row whose support differs from the
  oracle's at a near-threshold tie class.

Each is pinned here against something other than itself: the separately
pinned per-row functions (``linear_logp_row``, ``logp_row``), closed forms
written out by hand from the definition ("Configurable H100 consistency
runs", sampling-flags and KL-reference paragraphs), and exhaustive
enumeration on 16-token rows.  Planted mistakes at the end must each fail a
pin.
"""

import math

import numpy as np
import pytest

import oracle
from test_oracle_pins import V, VPAD, _brute_force, make_row

H = 8


def _bits(a):
    a = np.asarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


# ------------------------------------------------------ linear_logp_rows

def _lin_case(seed=31, n=4):
    rng = np.random.default_rng(seed)
    w = _bits(rng.standard_normal((VPAD, H)).astype(np.float32))
    w[V:] = 0x7FC0                      # NaN padding rows must be ignored
    h = _bits(rng.standard_normal((n, H)).astype(np.float32) * 1.5)
    targets = rng.integers(0, V, n)
    return h, w, targets


def pin_rows_equal_row_loop(impl):
    """Row by row equal to the pinned single-row function, with distinct
    per-row temperatures (a wrong tau index changes some row) and a scalar one."""
    h, w, tg = _lin_case()
    taus = np.array([0.7, 1.3, 0.5, 2.0], np.float32)
    got = impl(h, w, taus, tg)
    for i in range(h.shape[0]):
        want = oracle.linear_logp_row(h[i], w, float(taus[i]), int(tg[i]))
        assert abs(got[i] - want) < 1e-12, (i, got[i], want)
    got = impl(h, w, 0.9, tg)
    for i in range(h.shape[0]):
        want = oracle.linear_logp_row(h[i], w, 0.9, int(tg[i]))
        assert abs(got[i] - want) < 1e-12, i


def pin_rows_closed_forms(impl):
    """Row 0: zero hidden state gives -ln V; row 1: h = e_0 reduces to the
    logits oracle on weight column 0; row 2: h = 2 e_1 with tau 2 gives the
    same logits as h = e_1 with tau 1 (exact scaling by a power of two)."""
    rng = np.random.default_rng(32)
    w = _bits(3.0 * rng.standard_normal((VPAD, H)).astype(np.float32))
    h = np.zeros((4, H), np.uint16)
    h[1] = _bits([1.0] + [0.0] * (H - 1))
    h[2] = _bits([0.0, 2.0] + [0.0] * (H - 2))
    h[3] = _bits([0.0, 1.0] + [0.0] * (H - 2))
    tg = np.array([5, 777, 151935, 151935])
    got = impl(h, w, np.array([0.7, 1.0, 2.0, 1.0], np.float32), tg)
    assert abs(got[0] - (-math.log(V))) < 1e-12
    row = np.full(VPAD, 0xFF80, np.uint16)
    row[:V] = w[:V, 0]
    assert abs(got[1] - oracle.logp_row(row, 1.0, 1.0, -1, 777).full) < 1e-12
    assert abs(got[2] - got[3]) < 1e-12
    row[:V] = w[:V, 1]
    assert abs(got[3] - oracle.logp_row(row, 1.0, 1.0, -1, 151935).full) < 1e-12


LIN_ROWS_PINS = [pin_rows_equal_row_loop, pin_rows_closed_forms]


@pytest.mark.parametrize("pin", LIN_ROWS_PINS, ids=lambda f: f.__name__)
def test_linear_rows_pin(pin):
    pin(oracle.linear_logp_rows)


def _mut_rows_tau_shifted(h, w, tau, targets):
    """Mistake: the per-row temperature is taken from the next row."""
    if np.ndim(tau):
        tau = np.roll(np.asarray(tau), -1)
    return oracle.linear_logp_rows(h, w, tau, targets)


def _mut_rows_first_tau(h, w, tau, targets):
    """Mistake: the first row's temperature is used for every row."""
    t0 = float(np.asarray(tau).reshape(-1)[0])
    return oracle.linear_logp_rows(h, w, t0, targets)


def _mut_rows_target_shifted(h, w, tau, targets):
    """Mistake: the targets are read one row off."""
    return oracle.linear_logp_rows(h, w, tau, np.roll(np.asarray(targets), 1))


@pytest.mark.parametrize("mutant", [_mut_rows_tau_shifted, _mut_rows_first_tau,
                                    _mut_rows_target_shifted], ids=lambda f: f.__name__)
def test_planted_linear_rows_mistake_is_caught(mutant):
    failed = []
    for pin in LIN_ROWS_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"


# ------------------------------------------------------ row_logprobs_all

def _staircase():
    return make_row(-128.0, {j: -float(j) for j in range(64)})


def _two_valued():
    hot = list(range(1000, 1000 + 32 * 97, 97))
    return make_row(0.0, {j: 12.0 for j in hot}), hot


def _ties():
    return make_row(-20.0, {10: 3.0, 11: 2.0, 12: 1.0, 13: 1.0, 14: 1.0, 15: 1.0, 16: 1.0})


def pin_all_closed_forms(impl):
    """Closed forms on every token of the pinned rows.

    Staircase x_j = -j (j < 64), rest -128, tau 1, p 0.95: S = {0, 1, 2},
    restr_j = -j - ln(1 + e^-1 + e^-2) there; full_j = -j - ln Z.
    Two-valued row (32 hot at 12, tau 0.7, p 0.95): S = the hot set,
    restr = -ln 32 on it; full = closed form with the float32 quotient.
    Tie row (k = 3, ties at the third value): S = the 7 tokens >= 1.
    Uniform row: every token -ln V on both sides, S = everything.
    """
    full, restr, S = impl(_staircase(), 1.0, 0.95, -1)
    z = math.fsum([math.exp(-j) for j in range(64)] + [(V - 64) * math.exp(-128.0)])
    assert np.array_equal(np.nonzero(S)[0], [0, 1, 2])
    zs = 1 + math.exp(-1) + math.exp(-2)
    for j in range(3):
        assert abs(restr[j] - (-j - math.log(zs))) < 1e-12
    assert abs(restr[0] - (-0.4076059644443804)) < 1e-12
    assert np.all(restr[3:] == -np.inf)
    for j in (0, 1, 5, 63):
        assert abs(full[j] - (-j - math.log(z))) < 1e-12
    assert abs(full[0] - (-0.45867514538708193)) < 1e-12
    assert abs(full[100] - (-128.0 - math.log(z))) < 1e-9

    row, hot = _two_valued()
    full, restr, S = impl(row, 0.7, 0.95, -1)
    hs = float(np.float32(12.0) / np.float32(0.7))
    full_hot = -math.log(32 + (V - 32) * math.exp(-hs))
    assert np.array_equal(np.nonzero(S)[0], hot)
    assert np.all(np.abs(restr[hot] - (-math.log(32))) < 1e-12)
    assert np.sum(np.isfinite(restr)) == 32
    assert np.all(np.abs(full[hot] - full_hot) < 1e-12)
    assert abs(full[5] - (full_hot - hs)) < 1e-12

    full, restr, S = impl(_ties(), 1.0, 1.0, 3)
    assert np.array_equal(np.nonzero(S)[0], np.arange(10, 17))
    zs = math.exp(3) + math.exp(2) + 5 * math.exp(1)
    assert abs(restr[10] - (3 - math.log(zs))) < 1e-12
    assert abs(restr[16] - (1 - math.log(zs))) < 1e-12

    full, restr, S = impl(make_row(1.5), 1.3, 0.99, 128)
    assert S.all() and np.all(np.abs(full + math.log(V)) < 1e-12) and np.all(np.abs(restr + math.log(V)) < 1e-12)


def pin_all_brute_force_16(impl):
    """16 finite tokens among -inf: every token's full and restricted logprob
    and the support set against exhaustive enumeration over all 2^16 subsets."""
    rng = np.random.default_rng(16)
    cols = np.sort(rng.choice(V, 16, replace=False))
    for case in range(3):
        vals = (np.round(rng.standard_normal(16) * (2 + case)) / 2).astype(np.float32)
        row = make_row(float("-inf"), {int(c): float(v) for c, v in zip(cols, vals)})
        for tau, p, k in [(1.0, 0.9, -1), (0.7, 0.6, 5), (1.3, 1.0, 3), (2.0, 0.3, -1)]:
            bf_full, bf_restr, nS = _brute_force(vals, tau, p, k)
            full, restr, S = impl(row, tau, p, k)
            assert int(np.count_nonzero(S)) == nS
            assert np.all(S[cols] == np.isfinite(bf_restr))
            for i, c in enumerate(cols):
                assert abs(full[c] - bf_full[i]) < 1e-12
                assert (restr[c] == -math.inf and bf_restr[i] == -math.inf) or \
                    abs(restr[c] - bf_restr[i]) < 1e-12
            others = np.setdiff1d(np.arange(V), cols)[::997]
            assert np.all(full[others] == -np.inf) and np.all(restr[others] == -np.inf)


def pin_all_equals_logp_row(impl):
    """Equal to the pinned per-target function on every token of the small
    rows' finite columns and on a sample of the others, on a random spread row."""
    rng = np.random.default_rng(77)
    x = (3.0 * rng.standard_normal(VPAD)).astype(np.float32)
    spread = _bits(x)
    rows = [(_staircase(), 1.0, 0.95, -1, list(range(70))),
            (_ties(), 1.0, 0.8, 3, list(range(8, 20))),
            (spread, 0.7, 0.9, 500, list(np.argsort(-x[:V])[:40]) + list(rng.integers(0, V, 10)))]
    for row, tau, p, k, ts in rows:
        full, restr, S = impl(row, tau, p, k)
        for t in ts:
            r = oracle.logp_row(row, tau, p, k, int(t))
            assert abs(full[t] - r.full) < 1e-12 or (full[t] == r.full)
            assert (restr[t] == r.restr) or abs(restr[t] - r.restr) < 1e-12, (t, restr[t], r.restr)
        assert int(np.count_nonzero(S)) == oracle.logp_row(row, tau, p, k, 0).support


ALL_PINS = [pin_all_closed_forms, pin_all_brute_force_16, pin_all_equals_logp_row]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_row_logprobs_all_pin(pin):
    pin(oracle.row_logprobs_all)


def _mut_all_restr_over_full_z(row, tau, p, k):
    """Mistake: restricted logprobs normalised by the full mass, not Z_S."""
    full, restr, S = oracle.row_logprobs_all(row, tau, p, k)
    out = np.full_like(full, -np.inf)
    out[S] = full[S]
    return full, out, S


def _mut_all_topp_on_full(row, tau, p, k):
    """Mistake: top-p measured on the full distribution, then cut to S_k."""
    full, _, _ = oracle.row_logprobs_all(row, tau, p, -1)
    s = oracle.scaled_logits(row, tau)
    sk = oracle.top_k_mask(s, k)
    S = oracle.top_p_mask(s, np.ones_like(sk), p)[0] & sk if p < 1.0 else sk
    m = float(np.max(s))
    restr = np.full_like(s, -np.inf)
    restr[S] = (s[S] - m) - math.log(math.fsum(np.exp(s[S] - m)))
    return full, restr, S


def _mut_all_no_tau_full(row, tau, p, k):
    """Mistake: the full side drops the temperature."""
    _, restr, S = oracle.row_logprobs_all(row, tau, p, k)
    full, _, _ = oracle.row_logprobs_all(row, 1.0, p, k)
    return full, restr, S


@pytest.mark.parametrize("mutant", [_mut_all_restr_over_full_z, _mut_all_topp_on_full,
                                    _mut_all_no_tau_full], ids=lambda f: f.__name__)
def test_planted_row_logprobs_all_mistake_is_caught(mutant):
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"


# ------------------------------------------------------ restr_for_support_size

def pin_size_closed_forms(impl):
    """Staircase, tau 1: the top n tokens by value.  n = 3 gives the nucleus
    of p = 0.95 (-0.4076059644443804 at token 0); n = 2 gives -ln(1 + e^-1)
    at token 0 and -1 - ln(1 + e^-1) at token 1; n = 1 gives 0; a token
    outside the top n gives -inf.  Tie row: n = 7 keeps the whole class at 1."""
    row = _staircase()
    assert abs(impl(row, 1.0, 0, 3) - (-0.4076059644443804)) < 1e-12
    assert abs(impl(row, 1.0, 0, 2) - (-math.log1p(math.exp(-1)))) < 1e-12
    assert abs(impl(row, 1.0, 1, 2) - (-1 - math.log1p(math.exp(-1)))) < 1e-12
    assert impl(row, 1.0, 0, 1) == 0.0
    assert impl(row, 1.0, 2, 2) == -math.inf
    zs = math.exp(3) + math.exp(2) + 5 * math.exp(1)
    assert abs(impl(_ties(), 1.0, 14, 7) - (1 - math.log(zs))) < 1e-12


def pin_size_equals_oracle_support(impl):
    """With n = the oracle's own support size the value is logp_row's
    restricted logprob (top-p-only, top-k-only and combined rows)."""
    rng = np.random.default_rng(5)
    x = (2.0 * rng.standard_normal(VPAD)).astype(np.float32)
    row = _bits(x)
    top = np.argsort(-x[:V])
    for tau, p, k in [(0.7, 0.9, -1), (1.0, 1.0, 50), (1.3, 0.95, 300)]:
        r0 = oracle.logp_row(row, tau, p, k, int(top[0]))
        for t in (int(top[0]), int(top[3]), int(top[r0.support - 1])):
            want = oracle.logp_row(row, tau, p, k, t).restr
            assert abs(impl(row, tau, t, r0.support) - want) < 1e-12


def pin_size_rejects_tie_interior(impl):
    """n inside a tie class is not a support the definition can give."""
    with pytest.raises(AssertionError):
        impl(_ties(), 1.0, 10, 4)         # 3 tokens above the class of 5
    with pytest.raises(AssertionError):
        impl(make_row(1.5), 0.7, 0, 100)  # uniform row: one class of V


SIZE_PINS = [pin_size_closed_forms, pin_size_equals_oracle_support, pin_size_rejects_tie_interior]


@pytest.mark.parametrize("pin", SIZE_PINS, ids=lambda f: f.__name__)
def test_restr_for_support_size_pin(pin):
    pin(oracle.restr_for_support_size)


def _mut_size_off_by_one(row, tau, t, n):
    """Mistake: one token fewer than asked."""
    return oracle.restr_for_support_size(row, tau, t, n - 1) if n > 1 else 0.0


def _mut_size_full_normaliser(row, tau, t, n):
    """Mistake: normalised by the whole vocabulary's mass."""
    v = oracle.restr_for_support_size(row, tau, t, n)
    return v if v == -math.inf else oracle.logp_row(row, tau, 1.0, -1, t).full


def _mut_size_no_boundary_check(row, tau, t, n):
    """Mistake: a tie-class interior is accepted (ties broken by index)."""
    s = oracle.scaled_logits(row, tau)
    order = np.argsort(-s, kind="stable")[:n]
    if t not in order:
        return -math.inf
    m = float(np.max(s))
    return (float(s[t]) - m) - math.log(math.fsum(np.exp(s[order] - m)))


@pytest.mark.parametrize("mutant", [_mut_size_off_by_one, _mut_size_full_normaliser,
                                    _mut_size_no_boundary_check], ids=lambda f: f.__name__)
def test_planted_support_size_mistake_is_caught(mutant):
    failed = []
    for pin in SIZE_PINS:
        try:
            pin(mutant)
        except (AssertionError, pytest.fail.Exception):
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"
