"""Pins for the oracle's logprob gradient (CPU only).

Each pin checks ``oracle.logp_grad_row`` against something other than its
own formula: closed forms derived by hand, torch autograd (fp64) on the
forward definition with the support held fixed, and invariants of a softmax
gradient.  Planted mistakes at the end must each fail at least one pin.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import V, VPAD, fp32_quotient, make_row


def _grad(impl, row, tau, p, k, t, gf, gr):
    return impl(row, tau, p, k, t, gf, gr)


# --------------------------------------------------------------- pins

def pin_uniform(impl):
    """Uniform row: p_j = 1/V, so d full / d x_j = (1[j==t] - 1/V) / tau."""
    row = make_row(1.5)
    tau, t = 0.7, 5
    g = _grad(impl, row, tau, 1.0, -1, t, 1.0, 0.0)
    tau32 = float(np.float32(tau))
    assert abs(g[0] - (-1.0 / V / tau32)) < 1e-15
    assert abs(g[t] - (1.0 - 1.0 / V) / tau32) < 1e-12
    assert np.all(g[V:] == 0.0)


def pin_two_valued_restricted(impl):
    """32 tokens at 12, the rest at 0, tau 0.7, p 0.95: S = the 32 hot tokens
    (their mass is 0.99983), q = 1/32 on S, so d restr / d x_j = (1[j==t] - 1/32)/tau
    on S and 0 elsewhere; d full / d x_j follows from the two-valued softmax."""
    hot = list(range(1000, 1000 + 32 * 97, 97))
    row = make_row(0.0, {j: 12.0 for j in hot})
    tau = 0.7
    tau32 = float(np.float32(tau))
    t = hot[3]
    g = _grad(impl, row, tau, 0.95, -1, t, 0.0, 1.0)
    assert abs(g[t] - (1 - 1 / 32) / tau32) < 1e-12
    assert abs(g[hot[0]] - (-1 / 32) / tau32) < 1e-12
    assert g[0] == 0.0 and g[999] == 0.0
    # full side: p_hot = e^h / (32 e^h + V - 32) with h the float32 quotient 12/0.7
    h = fp32_quotient(12.0, 0.7)
    z = 32 * math.exp(h) + (V - 32)
    gf = _grad(impl, row, tau, 1.0, -1, t, 1.0, 0.0)
    assert abs(gf[t] - (1 - math.exp(h) / z) / tau32) < 1e-12
    assert abs(gf[0] - (-1 / z) / tau32) < 1e-15


def _autograd(bits_row, tau, p, k, t, gf, gr):
    """torch autograd, fp64, through s = x / tau with the support held fixed.
    s takes the float32 quotient's values (the operator's scaling) and the
    derivative 1/tau of the division."""
    x32 = oracle.bf16_bits_to_f32(bits_row[:V])
    x = torch.tensor(x32.astype(np.float64), requires_grad=True)
    s32 = torch.tensor((x32 / np.float32(tau)).astype(np.float64))
    s = s32 + (x - x.detach()) / float(np.float32(tau))
    full = s[t] - torch.logsumexp(s, 0)
    s_np = oracle.scaled_logits(bits_row, tau)
    sk = oracle.top_k_mask(s_np, k)
    S = oracle.top_p_mask(s_np, sk, p)[0] if p < 1.0 else sk
    loss = gf * full
    if S[t]:
        m = torch.as_tensor(S)
        restr = s[t] - torch.logsumexp(s[m], 0)
        loss = loss + gr * restr
    loss.backward()
    return x.grad.numpy()


def pin_autograd(impl):
    """Random rows (several tau / p / k): the oracle's gradient equals fp64
    autograd of the forward definition over all 151936 columns."""
    rng = np.random.default_rng(7)
    for tau, p, k, gf, gr in [(0.7, 0.9, 50, 1.0, 0.0), (1.3, 0.99, 128, 0.3, -1.7),
                              (1.0, 0.8, -1, -0.5, 2.0), (2.0, 1.0, 7, 0.0, 1.0)]:
        x = (2.0 * rng.standard_normal(V)).astype(np.float32)
        row = np.full(VPAD, 0xFF80, np.uint16)
        row[:V] = (x.view(np.uint32) >> 16).astype(np.uint16)
        s = oracle.scaled_logits(row, tau)
        t = int(np.argmax(s))          # the maximum is in every support
        want = _autograd(row, tau, p, k, t, gf, gr)
        got = _grad(impl, row, tau, p, k, t, gf, gr)
        assert np.allclose(got[:V], want, rtol=1e-9, atol=1e-15), (tau, p, k)
        assert np.all(got[V:] == 0.0)


def pin_invariants(impl):
    """A softmax gradient sums to zero over the row; outside the support the
    restricted part vanishes; a target outside S leaves only the full part."""
    rng = np.random.default_rng(8)
    x = (3.0 * rng.standard_normal(V)).astype(np.float32)
    row = np.full(VPAD, 0xFF80, np.uint16)
    row[:V] = (x.view(np.uint32) >> 16).astype(np.uint16)
    tau, p, k = 0.9, 0.9, 40
    s = oracle.scaled_logits(row, tau)
    t_in = int(np.argmax(s))
    g = _grad(impl, row, tau, p, k, t_in, 1.0, 1.0)
    assert abs(math.fsum(g)) < 1e-12
    sk = oracle.top_k_mask(s, k)
    S = oracle.top_p_mask(s, sk, p)[0]
    gr = _grad(impl, row, tau, p, k, t_in, 0.0, 1.0)
    assert np.all(gr[:V][~S] == 0.0) and abs(math.fsum(gr)) < 1e-12
    t_out = int(np.argmin(s))
    g_out = _grad(impl, row, tau, p, k, t_out, 0.0, 1.0)
    assert np.all(g_out == 0.0)
    assert np.array_equal(_grad(impl, row, tau, p, k, t_out, 1.0, 1.0),
                          _grad(impl, row, tau, p, k, t_out, 1.0, 0.0))


def pin_special_rows(impl):
    """Greedy rows have a zero gradient; NaN rows give NaN on the real columns;
    padded columns (whatever they hold) get 0."""
    row = make_row(-3.0, {10: 2.0}, pad="garbage")
    assert np.all(_grad(impl, row, 0.0, 1.0, -1, 10, 1.0, 1.0) == 0.0)
    g = _grad(impl, row, 1.0, 0.9, -1, 10, 1.0, 0.0)
    assert np.all(g[V:] == 0.0) and np.all(np.isfinite(g))
    bad = make_row(-3.0, {10: 2.0})
    bad[77] = 0x7FC0
    g = _grad(impl, bad, 1.0, 0.9, -1, 10, 1.0, 0.0)
    assert np.all(np.isnan(g[:V])) and np.all(g[V:] == 0.0)
    # a -inf target: full = -inf, its derivative is still 1/tau at t
    row = make_row(0.0, {3: float("-inf")})
    g = _grad(impl, row, 0.5, 1.0, -1, 3, 1.0, 0.0)
    assert abs(g[3] - 2.0) < 1e-15 and abs(g[0] - (-2.0 / (V - 1))) < 1e-15


GRAD_PINS = [pin_uniform, pin_two_valued_restricted, pin_autograd, pin_invariants, pin_special_rows]


@pytest.mark.parametrize("pin", GRAD_PINS, ids=lambda f: f.__name__)
def test_grad_pin(pin):
    pin(oracle.logp_grad_row)


# ------------------------------------------------------ planted mistakes

def _mut_no_tau(row, tau, p, k, t, gf, gr):
    return oracle.logp_grad_row(row, tau, p, k, t, gf, gr) * float(np.float32(tau))


def _mut_no_onehot(row, tau, p, k, t, gf, gr):
    g = oracle.logp_grad_row(row, tau, p, k, t, gf, gr)
    g[t] -= (gf + gr) / float(np.float32(tau)) if tau > 0 else 0.0
    return g


def _mut_restricted_as_full(row, tau, p, k, t, gf, gr):
    # mistake: the restricted part normalised over the whole vocabulary
    return oracle.logp_grad_row(row, tau, 1.0, -1, t, gf + gr, 0.0)


def _mut_shifted(row, tau, p, k, t, gf, gr):
    g = oracle.logp_grad_row(row, tau, p, k, t, gf, gr)
    g[:V] = np.roll(g[:V], 1)
    return g


def _mut_sign(row, tau, p, k, t, gf, gr):
    return -oracle.logp_grad_row(row, tau, p, k, t, gf, gr)


@pytest.mark.parametrize("mutant", [_mut_no_tau, _mut_no_onehot, _mut_restricted_as_full,
                                    _mut_shifted, _mut_sign], ids=lambda f: f.__name__)
def test_planted_gradient_mistake_is_caught(mutant):
    failed = []
    for pin in GRAD_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"
