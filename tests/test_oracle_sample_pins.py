"""Pins for the oracle's sampler and its random-bit generator (CPU only).

The generator is pinned by the known-answer vectors published with the
Philox4x32-10 definition; the sampler by closed-form draws on rows whose
restricted distribution is known by hand, and by stratified frequencies
checked against the (separately pinned) restricted logprobs of logp_row.
Planted mistakes at the end must each fail at least one pin.
"""

import math

import numpy as np
import pytest

import oracle
from test_oracle_pins import V, VPAD, make_row

# Known-answer vectors of Philox4x32-10 (counter words, key words, output words),
# as distributed with the Random123 library by the authors of "Parallel random
# numbers: as easy as 1, 2, 3" (SC 2011).
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def test_philox_known_answers():
    for ctr, key, want in PHILOX_KAT:
        assert oracle.philox4x32_10(ctr, key) == want


def test_philox_uniform_bits_layout():
    # seed low/high -> key words, counter low/high -> counter words 0/1
    seed, ctr = 0x299F31D0A4093822, 0x85A308D3243F6A88
    assert oracle.philox_uniform_bits(seed, ctr) == oracle.philox4x32_10(
        (0x243F6A88, 0x85A308D3, 0, 0), (0xA4093822, 0x299F31D0))[0]


def _u_mid(i, n):
    """32-bit draw in the middle of the i-th of n equal intervals of [0, 1)."""
    return int((i + 0.5) * 2 ** 32 / n)


# --------------------------------------------------------------- pins

def pin_two_valued(impl):
    """32 hot tokens at 12 (rest 0), tau 0.7, p 0.95: S = the hot tokens with
    equal mass, so U in [i/32, (i+1)/32) draws the i-th hot column in ascending
    order; its restricted logprob is -ln 32."""
    hot = sorted(range(1000, 1000 + 32 * 97, 97), reverse=True)
    row = make_row(0.0, {j: 12.0 for j in hot})
    cols = sorted(hot)
    for i in (0, 1, 17, 31):
        r = impl(row, 0.7, 0.95, -1, _u_mid(i, 32))
        assert r.token == cols[i], (i, r.token)
        assert abs(r.restr + math.log(32)) < 1e-12 and r.support == 32


def pin_staircase(impl):
    """x_j = -j on columns 0..63, rest -128, tau 1, p 0.95: S = {0, 1, 2} with
    masses 1, e^-1, e^-2; the edges of the CDF are 1/Z and (1 + e^-1)/Z."""
    row = make_row(-128.0, {j: -float(j) for j in range(64)})
    z = 1 + math.exp(-1) + math.exp(-2)
    e1, e2 = 1 / z, (1 + math.exp(-1)) / z
    cases = [(0.0, 0), (e1 - 1e-6, 0), (e1 + 1e-6, 1), (e2 - 1e-6, 1), (e2 + 1e-6, 2),
             (1 - 2 ** -32, 2)]
    for u, want in cases:
        r = impl(row, 1.0, 0.95, -1, int(u * 2 ** 32))
        assert r.token == want, (u, r.token)
    assert abs(impl(row, 1.0, 0.95, -1, 0).restr - (-math.log(z))) < 1e-12


def pin_stratified_frequencies(impl):
    """Stratified draws U = (i + 1/2)/N: each token is drawn N q_j times up to
    one, with q_j = exp(restr_j) from logp_row."""
    rng = np.random.default_rng(3)
    x = (2.0 * rng.standard_normal(V)).astype(np.float32)
    row = np.full(VPAD, 0xFF80, np.uint16)
    row[:V] = (x.view(np.uint32) >> 16).astype(np.uint16)
    tau, p, k = 0.8, 0.9, 60
    n = 256
    counts = {}
    for i in range(n):
        a = impl(row, tau, p, k, _u_mid(i, n)).token
        counts[a] = counts.get(a, 0) + 1
    _, restr, S = oracle.row_logprobs_all(row, tau, p, k)
    assert set(counts) <= set(np.nonzero(S)[0].tolist())
    for j in np.nonzero(S)[0]:
        assert abs(counts.get(int(j), 0) - n * math.exp(restr[j])) <= 1.0 + 1e-9, j


def pin_edges(impl):
    """Greedy rows and k = 1 give the argmax whatever U; U = 0 gives the lowest
    column of S; NaN rows give -1."""
    row = make_row(0.0, {500: 7.0, 90000: 7.0, 3: 6.0, 151935: 6.5})
    for u in (0, 2 ** 31, 2 ** 32 - 1):
        assert impl(row, 0.0, 1.0, -1, u).token == 500
        assert impl(row, 0.9, 1.0, 1, u).token in (500, 90000)
    r = impl(row, 1.0, 0.999, 4, 0)
    assert r.token == 3 and r.support == 4
    assert impl(row, 1.0, 0.999, 4, 2 ** 32 - 1).token == 151935
    bad = row.copy()
    bad[9] = 0x7FC0
    assert impl(bad, 1.0, 0.9, -1, 5).token == -1


SAMPLE_PINS = [pin_two_valued, pin_staircase, pin_edges, pin_stratified_frequencies]  # cheapest first


@pytest.mark.parametrize("pin", SAMPLE_PINS, ids=lambda f: f.__name__)
def test_sample_pin(pin):
    pin(oracle.sample_row)


# ------------------------------------------------------ planted mistakes

def _mut_value_order(row, tau, p, k, u):
    """Mistake: the CDF runs over the support in descending value order."""
    r = oracle.sample_row(row, tau, p, k, u)
    if r.token < 0 or tau == 0.0:
        return r
    s = oracle.scaled_logits(row, tau)
    _, restr, S = oracle.row_logprobs_all(row, tau, p, k)
    cols = np.nonzero(S)[0]
    order = cols[np.argsort(-s[cols], kind="stable")]
    cum = np.cumsum(np.exp(restr[order]))
    a = int(order[min(int(np.searchsorted(cum, u / 2 ** 32, side="right")), len(order) - 1)])
    return oracle.SampleResult(a, restr[a], r.full, r.support)


def _mut_full_distribution(row, tau, p, k, u):
    """Mistake: the draw ignores the top-k/top-p support."""
    return oracle.sample_row(row, tau, 1.0, -1, u)


def _mut_shift(row, tau, p, k, u):
    """Mistake: an off-by-one in the inverse CDF (the next column of S)."""
    r = oracle.sample_row(row, tau, p, k, u)
    if r.token < 0 or tau == 0.0:
        return r
    _, restr, S = oracle.row_logprobs_all(row, tau, p, k)
    cols = np.nonzero(S)[0]
    i = min(int(np.searchsorted(cols, r.token)) + 1, len(cols) - 1)
    return oracle.SampleResult(int(cols[i]), restr[cols[i]], r.full, r.support)


def _mut_u_flipped(row, tau, p, k, u):
    """Mistake: 1 - U instead of U."""
    return oracle.sample_row(row, tau, p, k, (2 ** 32 - 1) - int(u))


@pytest.mark.parametrize("mutant", [_mut_value_order, _mut_full_distribution, _mut_shift,
                                    _mut_u_flipped], ids=lambda f: f.__name__)
def test_planted_sampler_mistake_is_caught(mutant):
    failed = []
    for pin in SAMPLE_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
            break
    assert failed, f"{mutant.__name__} passed every pin"
