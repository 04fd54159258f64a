"""Pins for the oracle's restricted logprob straight from the LM head (CPU only).

linear_logp_pair_row must reduce to the pinned logits oracle (logp_row) when
the hidden state picks one weight column (the logits are then exactly the
column's bf16 values), keep every tied token on a uniform row, agree with an
fp64 torch restatement (topk + sort + cumulative sum), and with exhaustive
enumeration on 16 finite tokens.  Planted mistakes at the end must each fail
at least one pin.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import V, VPAD, _brute_force

H = 8


def _bits(a):
    a = np.asarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _column_row(rng, hot=40):
    x = (4.0 * rng.standard_normal(VPAD)).astype(np.float32)
    x[rng.choice(V, hot, replace=False)] += 12.0
    return _bits(x)


def pin_reduces_to_logits_oracle(impl):
    """h = e_0: the logits are W[:, 0]; with tau 1 and 0.5 (exact divisions)
    full, restricted and the support equal logp_row's on that column."""
    rng = np.random.default_rng(41)
    wb = np.zeros((VPAD, H), np.uint16)
    col = _column_row(rng)
    wb[:, 0] = col
    h = _bits([1.0] + [0.0] * (H - 1))
    row = col.copy()
    row[V:] = 0xFF80
    for tau, p, k, t in ((1.0, 0.9, -1, 5), (0.5, 0.95, 50, 77), (1.0, 1.0, 128, 1000),
                         (0.5, 0.7, 3, 151935), (1.0, 0.99, 128, 42)):
        want = oracle.logp_row(row, tau, p, k, t)
        got = impl(h, wb, tau, p, k, t)
        assert abs(got.full - want.full) < 1e-12, (tau, p, k)
        assert got.support == want.support, (tau, p, k, got.support, want.support)
        assert (got.restr == want.restr) or abs(got.restr - want.restr) < 1e-12, (tau, p, k)


def pin_uniform_keeps_every_tie(impl):
    """Zero weights: every logit is 0, every token tied: top-k and top-p keep all."""
    wb = np.zeros((VPAD, H), np.uint16)
    h = _bits(np.linspace(-1, 1, H))
    for p, k in ((0.5, 5), (0.9, -1), (1.0, 1)):
        r = impl(h, wb, 0.7, p, k, 123)
        assert abs(r.full + math.log(V)) < 1e-12 and abs(r.restr + math.log(V)) < 1e-12
        assert r.support == V


def pin_torch_fp64(impl):
    """Random h and W: the support from torch.topk and a sorted cumulative sum in fp64."""
    rng = np.random.default_rng(42)
    wb = _bits(0.5 * rng.standard_normal((VPAD, H)).astype(np.float32))
    h = _bits(rng.standard_normal(H) * 2)
    hf = torch.tensor(oracle.bf16_bits_to_f32(h).astype(np.float64))
    wf = torch.tensor(oracle.bf16_bits_to_f32(wb[:V]).astype(np.float64))
    for tau, p, k in ((1.3, 0.9, -1), (0.7, 0.95, 64), (1.0, 1.0, 10), (2.0, 0.5, 1000)):
        s = (wf @ hf) / float(np.float32(tau))
        keep = torch.ones(V, dtype=torch.bool)
        if 0 < k < V:
            keep = s >= torch.topk(s, k).values[-1]
        if p < 1.0:
            sv, order = torch.sort(torch.where(keep, s, torch.tensor(-math.inf, dtype=s.dtype)), descending=True)
            w = torch.exp(sv - sv[0])
            cum_before = torch.cumsum(w, 0) - w
            zk = w.sum()
            nuc = torch.zeros(V, dtype=torch.bool)
            nuc[order[cum_before / zk < p]] = True
            keep = keep & nuc
        n = int(keep.sum())
        t = int(torch.argmax(s))
        want = float(s[t] - torch.logsumexp(s[keep], 0))
        r = impl(h, wb, tau, p, k, t)
        assert r.support == n, (tau, p, k, r.support, n)
        assert abs(r.restr - want) < 1e-11, (tau, p, k)


def pin_brute_force_16(impl):
    """16 finite tokens of W[:, 0] far above the rest (-30000): every token's
    restricted logprob and the support against enumeration of all subsets."""
    rng = np.random.default_rng(43)
    cols = np.sort(rng.choice(V, 16, replace=False))
    for case in range(3):
        vals = (np.round(rng.standard_normal(16) * (2 + case)) / 2).astype(np.float32)
        col = np.full(VPAD, _bits([-30000.0])[0], np.uint16)
        col[cols] = _bits(vals)
        wb = np.zeros((VPAD, H), np.uint16)
        wb[:, 0] = col
        h = _bits([1.0] + [0.0] * (H - 1))
        for tau, p, k in ((1.0, 0.9, -1), (0.5, 0.6, 5), (1.0, 1.0, 3), (0.5, 0.95, 12)):
            _, bf_restr, nS = _brute_force(vals, tau, p, k)
            for i, c in enumerate(cols):
                r = impl(h, wb, tau, p, k, int(c))
                assert r.support == nS, (tau, p, k, r.support, nS)
                assert (r.restr == -math.inf and bf_restr[i] == -math.inf) or abs(r.restr - bf_restr[i]) < 1e-12


PAIR_PINS = [pin_reduces_to_logits_oracle, pin_uniform_keeps_every_tie, pin_torch_fp64, pin_brute_force_16]


@pytest.mark.parametrize("pin", PAIR_PINS, ids=lambda f: f.__name__)
def test_linear_pair_pin(pin):
    pin(oracle.linear_logp_pair_row)


# ------------------------------------------------------ planted mistakes

def _logits(h, w, tau):
    hf = oracle.bf16_bits_to_f32(h).astype(np.float64)
    wf = oracle.bf16_bits_to_f32(w[:V]).astype(np.float64)
    return (wf @ hf) / float(np.float32(tau))


def _finish(s, S, t, full):
    m = float(np.max(s))
    restr = (float(s[t]) - m) - math.log(math.fsum(np.exp(s[S] - m))) if S[t] else -math.inf
    return oracle.RowResult(full=full, restr=restr, support=int(np.count_nonzero(S)))


def _mut_topp_before_topk(h, w, tau, p, k, t):
    s = _logits(h, w, tau)
    full = oracle.linear_logp_row(h, w, tau, t)
    S = oracle.top_p_mask(s, np.ones(V, bool), p)[0] if p < 1 else np.ones(V, bool)
    return _finish(s, S & oracle.top_k_mask(s, k), t, full)


def _mut_exclusive_ties(h, w, tau, p, k, t):
    s = _logits(h, w, tau)
    full = oracle.linear_logp_row(h, w, tau, t)
    sk = np.ones(V, bool)
    if 0 < k < V:
        sk = np.zeros(V, bool)
        sk[np.argsort(-s, kind="stable")[:k]] = True
    S = oracle.top_p_mask(s, sk, p)[0] if p < 1 else sk
    return _finish(s, S, t, full)


def _mut_full_normaliser(h, w, tau, p, k, t):
    r = oracle.linear_logp_pair_row(h, w, tau, p, k, t)
    return oracle.RowResult(full=r.full, restr=r.full if r.restr > -math.inf else r.restr, support=r.support)


@pytest.mark.parametrize("mutant", [_mut_topp_before_topk, _mut_exclusive_ties, _mut_full_normaliser],
                         ids=lambda f: f.__name__)
def test_planted_linear_pair_mistake_is_caught(mutant):
    failed = []
    for pin in PAIR_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"


# ------------------------------------------------------ linear_logp_pair_rows

def pin_rows_equal_the_row_definition(rows_impl):
    """The batch form, with scalar and with per-row tau, top_p, top_k, equals
    linear_logp_pair_row (itself pinned above) row by row."""
    rng = np.random.default_rng(44)
    wb = _bits(0.5 * rng.standard_normal((VPAD, H)).astype(np.float32))
    hb = _bits(rng.standard_normal((5, H)) * 2)
    taus = np.array([0.7, 1.0, 1.3, 2.0, 0.5], np.float32)
    ps = np.array([0.9, 0.95, 1.0, 0.5, 0.99], np.float32)
    ks = np.array([-1, 50, 128, -1, 7])
    tg = np.array([3, 77, 1000, 151935, 42])
    for tau, p, k in ((taus, ps, ks), (1.3, 0.99, 128)):
        full, restr, sup = rows_impl(hb, wb, tau, p, k, tg)
        for i in range(5):
            at = (lambda v: v[i] if np.ndim(v) else v)
            r = oracle.linear_logp_pair_row(hb[i], wb, float(at(tau)), float(at(p)), int(at(k)), int(tg[i]))
            assert full[i] == r.full and sup[i] == r.support, (i, tau)
            assert restr[i] == r.restr, (i, tau)


def test_linear_pair_rows_pin():
    pin_rows_equal_the_row_definition(oracle.linear_logp_pair_rows)


def _mut_rows_tau_shift(h, w, tau, p, k, targets):
    t = np.roll(tau, 1) if np.ndim(tau) else tau
    return oracle.linear_logp_pair_rows(h, w, t, p, k, targets)


def _mut_rows_first_params(h, w, tau, p, k, targets):
    first = (lambda v: v[0] if np.ndim(v) else v)
    return oracle.linear_logp_pair_rows(h, w, first(tau), first(p), first(k), targets)


def _mut_rows_target_roll(h, w, tau, p, k, targets):
    return oracle.linear_logp_pair_rows(h, w, tau, p, k, np.roll(np.asarray(targets), 1))


@pytest.mark.parametrize("mutant", [_mut_rows_tau_shift, _mut_rows_first_params, _mut_rows_target_roll],
                         ids=lambda f: f.__name__)
def test_planted_pair_rows_mistake_is_caught(mutant):
    with pytest.raises(AssertionError):
        pin_rows_equal_the_row_definition(mutant)
