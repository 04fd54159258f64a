"""CPU: the row-by-row comparison the GPU parity tests use, and its worker pool.

The "GPU outputs" here are made on the CPU from the oracle itself (plus
deviations planted on purpose), so these tests check the comparison logic:
that it passes outputs within the tolerance, fails a planted deviation and
names its row, counts a support that differs only at a tie class within
1e-6 of the nucleus threshold instead of failing it, and that the targets
drawn on the pool do not depend on the chunking.
"""

import math

import numpy as np
import pytest

import oracle
import _oracle_check as oc
from test_oracle_pins import make_row

V = oracle.VREAL


def _rows(n, seed):
    rng = np.random.default_rng(seed)
    x = (3.0 * rng.standard_normal((n, oracle.VPAD))).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    taus = rng.choice([0.0, 0.7, 1.3], n).astype(np.float32)
    ps = rng.choice([0.9, 0.95, 1.0], n).astype(np.float32)
    ks = rng.choice([-1, 20, 128], n).astype(np.int32)
    return bits, taus, ps, ks


def _oracle_outputs(bits, taus, ps, ks, ts):
    return oracle.logp_batch(bits, taus, ps, ks, ts)


def test_parallel_check_passes_and_catches_a_planted_deviation():
    bits, taus, ps, ks = _rows(40, 1)
    ts = oc.oracle_targets_parallel(bits, taus, ps, ks, np.arange(40) % 9 == 0, seed=5)
    full, restr, sup = _oracle_outputs(bits, taus, ps, ks, ts)
    full32, restr32 = full.astype(np.float32), restr.astype(np.float32)
    st = oc.Stats()
    oc.check_rows_parallel(st, bits, taus, ps, ks, ts, full32, restr32, sup)
    assert st.rows == 40 and st.support_differs == 0
    assert st.max_full <= 2e-6 and st.max_restr <= 2e-6
    bad = restr32.copy()
    i = int(np.nonzero(np.isfinite(restr32) & (taus > 0))[0][3])
    bad[i] += 1e-4
    with pytest.raises(AssertionError, match=f"row {i}:"):
        oc.check_rows_parallel(oc.Stats(), bits, taus, ps, ks, ts, full32, bad, sup)
    wrong_sup = sup.copy()
    j = int(np.nonzero((ps < 1) & (taus > 0))[0][0])
    wrong_sup[j] += 1
    with pytest.raises(AssertionError, match=f"row {j}:"):
        oc.check_rows_parallel(oc.Stats(), bits, taus, ps, ks, ts, full32, restr32, wrong_sup)


def test_kl_mode_checks_reference_and_difference():
    bits, _, _, _ = _rows(6, 2)
    rbits = bits.copy()
    rbits[:, :100] ^= 1                     # a nearby reference row
    ts = np.arange(6, dtype=np.int32) * 1000
    full, restr, sup = _oracle_outputs(bits, 1.3, 0.99, 128, ts)
    fref, _, _ = _oracle_outputs(rbits, 1.3, 1.0, -1, ts)
    kl = (full - fref).astype(np.float32)
    st = oc.Stats()
    oc.check_rows_parallel(st, bits, 1.3, 0.99, 128, ts, full, restr, sup, ref_bits=rbits,
                           full_ref=fref, kl=kl)
    assert st.rows == 6 and st.max_kl < 1e-6
    kl[2] += 1e-3
    with pytest.raises(AssertionError, match="kl"):
        oc.check_rows_parallel(oc.Stats(), bits, 1.3, 0.99, 128, ts, full, restr, sup,
                               ref_bits=rbits, full_ref=fref, kl=kl)


def test_near_threshold_support_is_counted_not_failed():
    """Staircase row with p set to the float32 value of a class's G: the two
    supports on either side of that class are both accepted and counted."""
    row = make_row(-128.0, {j: -float(j) for j in range(64)})
    r = oracle.logp_row(row, 1.0, 0.95, -1, 0, want_margins=True)
    p = float(np.float32(r.g_desc[3]))       # G of the 4th class, rounded to float32
    assert abs(p - r.g_desc[3]) / p <= oc.MARGIN
    o = oracle.logp_row(row, 1.0, p, -1, 0, want_margins=True)
    other = 4 if o.support == 3 else 3
    gpu_restr = oracle.restr_for_support_size(row, 1.0, 0, other)
    st = oc.Stats()
    oc.check_row(st, row, 1.0, p, -1, 0, o.full, gpu_restr, other)
    assert st.support_differs == 1 and st.near_rows == 1 and st.near_tokens >= 1
    # a support two classes away is not near the threshold: it fails
    with pytest.raises(AssertionError, match="margin"):
        oc.check_row(oc.Stats(), row, 1.0, p, -1, 0, o.full, gpu_restr, other + 2 if other == 4 else 2)


def test_targets_do_not_depend_on_chunking():
    bits, taus, ps, ks = _rows(20, 3)
    forced = np.arange(20) % 5 == 1
    a = oc.oracle_targets_parallel(bits, taus, ps, ks, forced, seed=9)
    b = np.array([oc.target_row(bits[i], float(taus[i]), float(ps[i]), int(ks[i]), bool(forced[i]),
                                (9, i)) for i in range(20)])
    assert np.array_equal(a, b)
    for i in range(20):
        o = oracle.logp_row(bits[i], float(taus[i]), float(ps[i]), int(ks[i]), int(a[i]))
        if forced[i] and o.support < V:
            assert o.restr == -math.inf
        elif not forced[i]:
            assert o.restr > -math.inf


def test_scaled_tolerance_term():
    """scale_tol widens the bound by scale_tol * max(|M|, |x_t|) / tau: on a
    row whose maximum is 24 at temperature 1e-3 (scaled logits of 24000) a
    deviation of 4e-3 passes with 2.4e-7 (bound 5.8e-3) and fails without;
    at temperature 1 the same term adds only 5.8e-6."""
    row = make_row(0.0, {3: 24.0, 9: 23.0})
    assert abs(oc.scaled_magnitude(row, 1e-3, 9) - 24.0 / float(np.float32(1e-3))) < 1e-6
    assert oc.scaled_magnitude(row, 0.0, 9) == 0.0
    r = oracle.logp_row(row, 1e-3, 1.0, -1, 9)
    st = oc.Stats()
    oc.check_row(st, row, 1e-3, 1.0, -1, 9, r.full + 4e-3, r.restr + 4e-3, r.support, scale_tol=2.4e-7)
    with pytest.raises(AssertionError):
        oc.check_row(oc.Stats(), row, 1e-3, 1.0, -1, 9, r.full + 4e-3, r.restr + 4e-3, r.support)
    r1 = oracle.logp_row(row, 1.0, 1.0, -1, 9)
    with pytest.raises(AssertionError):
        oc.check_row(oc.Stats(), row, 1.0, 1.0, -1, 9, r1.full + 4e-5, r1.restr, r1.support,
                     scale_tol=2.4e-7)
