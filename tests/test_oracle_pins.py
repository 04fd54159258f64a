"""Pins for the CPU oracle: closed forms, invariants, brute force and special cases.

Each pin checks the oracle against something other than itself: a value
derived by hand from the definition, a library routine for a special case,
or exhaustive enumeration on a tiny vocabulary.  The mutation tests at the
end plant plausible mistakes in the oracle and check that a pin catches
each of them.
"""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import logp_oracle as lo

V = oracle.VREAL
VPAD = oracle.VPAD
NEG_INF_BITS = 0xFF80


def f32_to_bf16_bits_exact(vals) -> np.ndarray:
    a = np.asarray(vals, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def make_row(fill: float, values: dict | None = None, pad="neginf") -> np.ndarray:
    row = np.empty(VPAD, dtype=np.uint16)
    row[:V] = f32_to_bf16_bits_exact([fill])[0]
    if pad == "neginf":
        row[V:] = NEG_INF_BITS
    elif pad == "garbage":
        row[V:] = f32_to_bf16_bits_exact([8192.0 if i % 3 else 0.0 for i in range(VPAD - V)])
        row[V::5] = 0x7FC0   # NaN
        row[V + 1::7] = 0x7F80  # +inf
    if values:
        idx = np.fromiter(values.keys(), dtype=np.int64)
        row[idx] = f32_to_bf16_bits_exact(list(values.values()))
    return row


def fp32_quotient(a: float, b: float) -> float:
    """Correctly rounded float32 quotient from exact rationals (independent of numpy's division)."""
    q = Fraction(float(np.float32(a))) / Fraction(float(np.float32(b)))
    return float(np.float32(float(q)))


# --------------------------------------------------------------- pin suite

def pin_uniform(impl):
    """Uniform logits: every token has logprob -ln(151936) on both sides."""
    row = make_row(1.5)
    want = -math.log(V)
    assert abs(want - (-11.931214658529285)) < 1e-15
    for tau, p, k, t in [(0.7, 0.95, -1, 0), (1.3, 0.99, 128, V - 1), (1.0, 1.0, -1, 12345)]:
        r = impl(row, tau, p, k, t)
        assert abs(r.full - want) < 1e-12
        assert abs(r.restr - want) < 1e-12     # all tokens tie: top-k and top-p keep all
        assert r.support == V


def pin_dominant(impl):
    """One logit at 64, the rest at -64, tau 1: the dominant token has logprob ~0."""
    row = make_row(-64.0, {77: 64.0})
    r = impl(row, 1.0, 0.95, -1, 77)
    assert abs(r.full - (-math.log1p((V - 1) * math.exp(-128.0)))) < 1e-45
    assert r.restr == 0.0 and r.support == 1
    r = impl(row, 1.0, 1.0, -1, 78)
    assert abs(r.full - (-128.0 - math.log1p((V - 1) * math.exp(-128.0)))) < 1e-12


def pin_topk1(impl):
    """top-k = 1 keeps only the (unique) argmax: logprob 0 there, -inf elsewhere."""
    rng = np.random.default_rng(11)
    vals = {int(j): float(v) for j, v in zip(rng.choice(V, 50, replace=False),
                                              np.arange(1, 51, dtype=np.float32))}
    row = make_row(0.0, vals)
    amax = max(vals, key=vals.get)
    for p in (1.0, 0.5):
        assert impl(row, 0.9, p, 1, amax).restr == 0.0
        r = impl(row, 0.9, p, 1, (amax + 1) % V)
        assert r.restr == -math.inf and r.support == 1


def pin_disabled_equals_full(impl):
    """p = 1 and k = -1 (or k = V) disable both filters: restricted == full exactly."""
    rng = np.random.default_rng(5)
    x = (3.0 * rng.standard_normal(VPAD)).astype(np.float32)
    row = (x.view(np.uint32) >> 16).astype(np.uint16)
    for k in (-1, V):
        r = impl(row, 0.8, 1.0, k, 4242)
        assert r.restr == r.full and r.support == V


def pin_two_valued(impl):
    """32 hot tokens at 12, the rest at 0, tau 0.7 (closed form with the fp32 quotient)."""
    n, h, tau = 32, 12.0, 0.7
    hot = list(range(1000, 1000 + 32 * 97, 97))
    row = make_row(0.0, {j: h for j in hot})
    hs = fp32_quotient(h, tau)
    full_hot = -math.log(n + (V - n) * math.exp(-hs))
    assert abs(full_hot - (-3.4659062495997226)) < 1e-6   # exact-12/0.7 value, for reference
    r = impl(row, tau, 0.95, -1, hot[3])
    assert abs(r.full - full_hot) < 1e-12
    assert abs(r.restr - (-math.log(32))) < 1e-12 and r.support == 32
    r = impl(row, tau, 0.95, -1, 5)
    assert abs(r.full - (-hs + full_hot)) < 1e-12 and r.restr == -math.inf


def pin_staircase(impl):
    """x_j = -j (j < 64), rest -128, tau 1, p 0.95: the nucleus is the top 3 tokens."""
    row = make_row(-128.0, {j: -float(j) for j in range(64)})
    z = math.fsum([math.exp(-j) for j in range(64)] + [(V - 64) * math.exp(-128.0)])
    r = impl(row, 1.0, 0.95, -1, 0)
    assert r.support == 3
    assert abs(r.restr - (-math.log(1 + math.exp(-1) + math.exp(-2)))) < 1e-12
    assert abs(r.restr - (-0.4076059644443804)) < 1e-12
    assert abs(r.full - (-math.log(z))) < 1e-12
    assert abs(r.full - (-0.45867514538708193)) < 1e-12
    assert abs(impl(row, 1.0, 0.95, -1, 2).restr - (-2 - math.log(1 + math.exp(-1) + math.exp(-2)))) < 1e-12
    assert impl(row, 1.0, 0.95, -1, 3).restr == -math.inf


def pin_order_topk_then_topp(impl):
    """k = 2 then p = 0.7 renormalised over the top 2: token 1 has G = 1/(1+e^-1) = 0.731 >= 0.7.

    Applying top-p first (on the full distribution, G = 0.632) would keep it.
    """
    row = make_row(-128.0, {j: -float(j) for j in range(64)})
    r = impl(row, 1.0, 0.7, 2, 0)
    assert r.support == 1 and r.restr == 0.0
    r = impl(row, 1.0, 0.75, 2, 1)
    assert r.support == 2 and abs(r.restr - (-1 - math.log(1 + math.exp(-1)))) < 1e-12


def pin_topk_ties(impl):
    """Ties at the k-th value are kept: 5 tokens share the 3rd largest value."""
    row = make_row(-20.0, {10: 3.0, 11: 2.0, 12: 1.0, 13: 1.0, 14: 1.0, 15: 1.0, 16: 1.0})
    r = impl(row, 1.0, 1.0, 3, 16)
    assert r.support == 7
    zs = math.exp(3) + math.exp(2) + 5 * math.exp(1)
    assert abs(r.restr - (1 - math.log(zs))) < 1e-12


def pin_greedy(impl):
    """tau 0: logprob 0 at the argmax (lowest index among ties), -inf elsewhere."""
    row = make_row(0.0, {500: 7.0, 90000: 7.0, 3: 6.0})
    r = impl(row, 0.0, 0.9, 50, 500)
    assert r.full == 0.0 and r.restr == 0.0 and r.support == 1
    r = impl(row, 0.0, 0.9, 50, 90000)
    assert r.full == -math.inf and r.restr == -math.inf


def pin_padding_and_nonfinite(impl):
    """Padded columns are ignored; NaN/+inf among real columns gives NaN; -inf is mass 0."""
    base = {j: float(j % 13) for j in range(0, V, 1237)}
    a = impl(make_row(-3.0, base, pad="neginf"), 0.9, 0.9, 64, 1237)
    b = impl(make_row(-3.0, base, pad="garbage"), 0.9, 0.9, 64, 1237)
    assert a.full == b.full and a.restr == b.restr and a.support == b.support
    row = make_row(-3.0, base)
    row[777] = 0x7FC0
    assert math.isnan(impl(row, 0.9, 0.9, 64, 1237).full)
    row[777] = 0x7F80
    assert math.isnan(impl(row, 0.9, 0.9, 64, 1237).restr)
    row = make_row(float("-inf"), {})
    assert math.isnan(impl(row, 1.0, 1.0, -1, 0).full)
    # -inf tokens carry no mass: a row of 2 finite tokens among -inf
    row = make_row(float("-inf"), {7: 0.0, 8: 0.0})
    r = impl(row, 1.0, 1.0, -1, 7)
    assert abs(r.full - (-math.log(2))) < 1e-15
    assert impl(row, 1.0, 1.0, -1, 9).full == -math.inf


def pin_invariants(impl):
    """Both distributions sum to one over their supports (40 finite tokens, rest -inf)."""
    rng = np.random.default_rng(21)
    cols = rng.choice(V, 40, replace=False)
    vals = np.round(rng.standard_normal(40) * 8) / 4      # exact in bf16, with ties
    row = make_row(float("-inf"), {int(c): float(v) for c, v in zip(cols, vals)})
    for tau, p, k in [(0.7, 0.9, -1), (1.3, 0.5, 10), (1.0, 1.0, 7), (2.0, 0.99, 30)]:
        res = [impl(row, tau, p, k, int(c)) for c in cols]
        assert abs(math.fsum(math.exp(r.full) for r in res) - 1.0) < 1e-12
        assert abs(math.fsum(math.exp(r.restr) for r in res) - 1.0) < 1e-12
        n_in = sum(r.restr > -math.inf for r in res)
        assert n_in == res[0].support


def _brute_force(xs16: np.ndarray, tau: float, p: float, k: int):
    """Enumerate every subset of 16 tokens (the definition read as sets):

    S_k = the smallest subset closed upward and under ties with |S_k| >= k;
    S   = the smallest-mass subset of S_k, closed upward and under ties,
          whose mass is >= p * mass(S_k).
    """
    s = (xs16.astype(np.float32) / np.float32(tau)).astype(np.float64)
    n = len(s)
    m = max(s)
    w = [math.exp(v - m) for v in s]

    def closed(mask):
        inside = [i for i in range(n) if mask >> i & 1]
        outside = [i for i in range(n) if not mask >> i & 1]
        return all(s[o] < s[i] for i in inside for o in outside)

    closed_sets = [mk for mk in range(1, 1 << n) if closed(mk)]
    size = lambda mk: bin(mk).count("1")
    mass = lambda mk: math.fsum(w[i] for i in range(n) if mk >> i & 1)
    if k == -1 or k >= n:
        sk = (1 << n) - 1
    else:
        sk = min((mk for mk in closed_sets if size(mk) >= k), key=size)
    if p >= 1.0:
        S = sk
    else:
        zk = mass(sk)
        S = min((mk for mk in closed_sets if (mk & ~sk) == 0 and mass(mk) >= p * zk), key=mass)
    lse_full = m + math.log(math.fsum(w))
    lse_S = m + math.log(mass(S))
    full = [s[i] - lse_full for i in range(n)]
    restr = [s[i] - lse_S if S >> i & 1 else -math.inf for i in range(n)]
    return full, restr, size(S)


def pin_brute_force_16(impl):
    rng = np.random.default_rng(16)
    cols = np.sort(rng.choice(V, 16, replace=False))
    for case in range(6):
        vals = (np.round(rng.standard_normal(16) * (2 + case)) / 2).astype(np.float32)
        row = make_row(float("-inf"), {int(c): float(v) for c, v in zip(cols, vals)})
        for tau, p, k in [(1.0, 0.9, -1), (0.7, 0.6, 5), (1.3, 1.0, 3), (0.5, 0.95, 12),
                          (2.0, 0.3, -1)]:
            full, restr, nS = _brute_force(vals, tau, p, k)
            for i, c in enumerate(cols):
                r = impl(row, tau, p, k, int(c))
                assert abs(r.full - full[i]) < 1e-12
                assert (r.restr == -math.inf and restr[i] == -math.inf) or abs(r.restr - restr[i]) < 1e-12
                assert r.support == nS


def pin_logsumexp_library(impl):
    """Special case: with both filters off, full = s_t - torch.logsumexp(s) in fp64."""
    rng = np.random.default_rng(9)
    x = (4 * rng.standard_normal(VPAD) + 2).astype(np.float32)
    row = (x.view(np.uint32) >> 16).astype(np.uint16)
    xb = torch.from_numpy(oracle.bf16_bits_to_f32(row[:V]).copy())
    s = (xb / torch.tensor(1.3, dtype=torch.float32)).double()
    lse = torch.logsumexp(s, 0).item()
    for t in (0, 100, V - 1):
        r = impl(row, 1.3, 1.0, -1, t)
        assert abs(r.full - (s[t].item() - lse)) < 1e-11


PINS = [pin_uniform, pin_dominant, pin_topk1, pin_disabled_equals_full, pin_two_valued,
        pin_staircase, pin_order_topk_then_topp, pin_topk_ties, pin_greedy,
        pin_padding_and_nonfinite, pin_invariants, pin_brute_force_16, pin_logsumexp_library]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.logp_row)


def test_fp32_scaling_is_float32_division():
    """The oracle's scaling equals the correctly rounded float32 quotient."""
    rng = np.random.default_rng(3)
    x = (6 * rng.standard_normal(4000)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    row = np.full(VPAD, NEG_INF_BITS, dtype=np.uint16)
    row[:4000] = bits
    for tau in (0.7, 1.3, 0.3):
        s = oracle.scaled_logits(row, tau)[:4000]
        want = [fp32_quotient(float(v), tau) for v in oracle.bf16_bits_to_f32(bits)]
        assert np.array_equal(s, np.asarray(want))


def test_shard_summaries_merge_to_global_lse():
    """Eight fixed shard (max, sum-exp) summaries merged in order equal the global LSE."""
    rng = np.random.default_rng(8)
    x = (3 * rng.standard_normal(VPAD)).astype(np.float32)
    x[19072 * 3 + 5] = 40.0       # the max sits in shard 3
    row = (x.view(np.uint32) >> 16).astype(np.uint16)
    row[V:] = 0x7F80                # +inf in padding must be ignored
    m, l = oracle.shard_summaries(row, 0.9)
    assert np.argmax(m) == 3
    s = torch.from_numpy(oracle.scaled_logits(row, 0.9))
    assert abs(oracle.merge_summaries(m, l) - torch.logsumexp(s, 0).item()) < 1e-11
    # shard 7 holds 18432 real and 640 padded columns
    assert oracle.SHARD_W * 7 + 18432 == V


def test_validation_rejects_out_of_domain():
    row = make_row(0.0)
    for args in [(-0.1, 0.9, -1, 0), (math.nan, 0.9, -1, 0), (math.inf, 0.9, -1, 0),
                 (1.0, 0.0, -1, 0), (1.0, 1.01, -1, 0), (1.0, math.nan, -1, 0),
                 (1.0, 0.9, 0, 0), (1.0, 0.9, -2, 0), (1.0, 0.9, V + 1, 0),
                 (1.0, 0.9, -1, -1), (1.0, 0.9, -1, V)]:
        with pytest.raises(oracle.InvalidArgument):
            oracle.logp_row(row, *args)
    full, restr, sup = oracle.logp_batch(np.stack([row, row]), 1.0, np.array([0.9, 2.0]), -1, 0)
    assert sup[1] == -1 and math.isnan(full[1]) and sup[0] == V


# ------------------------------------------------------ planted mistakes

def _fails_some_pin(monkeypatch_ctx) -> list:
    failed = []
    for pin in PINS:
        try:
            pin(oracle.logp_row)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    return failed


def _mut_topk_exclusive(s, top_k):
    n = s.shape[0]
    if top_k == -1 or top_k >= n:
        return np.ones(n, dtype=bool)
    keep = np.zeros(n, dtype=bool)
    keep[np.argsort(-s, kind="stable")[:top_k]] = True
    return keep


def _mut_topp_inclusive(s, sk, top_p):
    mask, uniq, counts, g = lo.__dict__["_orig_top_p_mask"](s, sk, top_p)
    # off by one class: use the mass at-or-above instead of strictly above
    m = np.max(s)
    vals = s[sk]
    z = math.fsum(np.exp(vals - m))
    at_or_above = np.cumsum(counts * np.exp(uniq - m)) / z
    keep_vals = uniq[at_or_above < top_p]
    new = sk & np.isin(s, keep_vals)
    return new, uniq, counts, g


def _mut_topp_first(s, sk, top_p):
    full_sk = np.ones_like(sk)
    mask = lo.__dict__["_orig_top_p_mask"](s, full_sk, top_p)[0]
    return mask & sk, None, None, None


def _mut_no_temperature(bits_row, tau, vreal=V):
    return lo.__dict__["_orig_scaled_logits"](bits_row, 1.0 if tau > 0 else tau, vreal)



def _mut_multiply_inverse(bits_row, tau, vreal=V):
    x = oracle.bf16_bits_to_f32(bits_row[:vreal])
    return (x * (np.float32(1.0) / np.float32(tau))).astype(np.float64)


MUTANTS = {
    "topk_exclusive_ties": ("top_k_mask", _mut_topk_exclusive),
    "topp_own_class_counted": ("top_p_mask", _mut_topp_inclusive),
    "topp_before_topk": ("top_p_mask", _mut_topp_first),
    "temperature_dropped": ("scaled_logits", _mut_no_temperature),
    "scaling_perturbed": ("scaled_logits", _mut_multiply_inverse),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setitem(lo.__dict__, "_orig_" + attr, getattr(lo, attr))
    monkeypatch.setattr(lo, attr, fn)
    failed = _fails_some_pin(monkeypatch)
    assert failed, f"mutant {name} passed every pin"


def test_planted_mistake_padding_included(monkeypatch):
    orig = lo.bf16_bits_to_f32

    def leaky_logp_row(bits_row, tau, top_p, top_k, target, vreal=V, want_margins=False):
        # mistake: the real-vocabulary cut is dropped (padded columns join the softmax)
        b = np.asarray(bits_row, dtype=np.uint16)
        return lo.__dict__["_orig_logp_row"](b, tau, top_p, top_k, target, vreal=VPAD)

    monkeypatch.setitem(lo.__dict__, "_orig_logp_row", lo.logp_row)
    monkeypatch.setattr(oracle, "logp_row", leaky_logp_row)
    failed = _fails_some_pin(monkeypatch)
    assert failed
    assert lo.bf16_bits_to_f32 is orig


def test_planted_mistake_greedy_last_index(monkeypatch):
    orig_argmax = np.argmax

    def last_argmax(a, *args, **kw):
        a = np.asarray(a)
        return a.shape[0] - 1 - orig_argmax(a[::-1], *args, **kw)

    monkeypatch.setattr(lo.np, "argmax", last_argmax)
    with pytest.raises(AssertionError):
        pin_greedy(oracle.logp_row)


def test_golden_tiny16_matches_brute_force():
    """The stored 16-token fixture agrees with exhaustive enumeration (and the oracle)."""
    import json, os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny16.json")
    data = json.load(open(path))
    dec = lambda v: -math.inf if v == "-inf" else float(v)
    for case in data["cases"]:
        vals = np.asarray(case["values"], dtype=np.float32)
        tau, p, k = case["tau"], case["top_p"], case["top_k"]
        if tau == 0.0:
            amax = int(np.argmax(vals))
            for i, (t, full, restr, sup) in enumerate(case["per_target"]):
                want = 0.0 if i == amax else -math.inf
                assert dec(full) == want and dec(restr) == want and sup == 1
            continue
        full_bf, restr_bf, nS = _brute_force(vals, tau, p, k)
        for i, (t, full, restr, sup) in enumerate(case["per_target"]):
            assert abs(dec(full) - full_bf[i]) < 1e-12
            assert dec(restr) == restr_bf[i] or abs(dec(restr) - restr_bf[i]) < 1e-12
            assert sup == (nS if (p < 1 or k != -1) else oracle.VREAL)
