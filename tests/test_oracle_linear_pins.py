"""Pins for the oracle's fused LM-head logprob (CPU only).

linear_logp_row must reduce to the (separately pinned) logits oracle when the
hidden state picks one weight column, give -ln V for zero weights, agree
with fp64 torch matmul + log-softmax, and ignore the padded weight rows.
Planted mistakes at the end must each fail at least one pin.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import V, VPAD

H = 8


def _bits(a):
    a = np.asarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _rand_w(rng, scale=1.0, pad=None):
    w = (scale * rng.standard_normal((VPAD, H))).astype(np.float32)
    wb = _bits(w)
    if pad is not None:
        wb[V:] = pad
    return wb


def pin_reduces_to_logits_oracle(impl):
    """h = e_0: the logits are W[:, 0]; with tau = 1 and 0.5 (exact divisions)
    the result equals logp_row's full logprob on those logits."""
    rng = np.random.default_rng(1)
    wb = _rand_w(rng, 3.0)
    h = _bits([1.0] + [0.0] * (H - 1))
    row = np.full(VPAD, 0xFF80, np.uint16)
    row[:V] = wb[:V, 0]
    for tau, t in ((1.0, 17), (0.5, 123456)):
        want = oracle.logp_row(row, tau, 1.0, -1, t).full
        assert abs(impl(h, wb, tau, t) - want) < 1e-12, tau


def pin_zero_weights(impl):
    wb = np.zeros((VPAD, H), np.uint16)
    h = _bits(np.linspace(-1, 1, H))
    assert abs(impl(h, wb, 0.7, 5) - (-math.log(V))) < 1e-12


def pin_torch_fp64(impl):
    """Random h and W: fp64 torch matmul and log-softmax over the real rows."""
    rng = np.random.default_rng(2)
    wb = _rand_w(rng, 0.5)
    h = _bits(rng.standard_normal(H))
    hf = torch.tensor(oracle.bf16_bits_to_f32(h).astype(np.float64))
    wf = torch.tensor(oracle.bf16_bits_to_f32(wb[:V]).astype(np.float64))
    for tau, t in ((1.3, 42), (0.6, 151935)):
        lp = torch.log_softmax((wf @ hf) / float(np.float32(tau)), 0)
        assert abs(impl(h, wb, tau, t) - float(lp[t])) < 1e-11, tau


def pin_padding_ignored(impl):
    rng = np.random.default_rng(3)
    w = _rand_w(rng)
    h = _bits(rng.standard_normal(H))
    a = impl(h, np.where(np.arange(VPAD)[:, None] < V, w, 0).astype(np.uint16), 1.0, 9)
    for pad in (0x4680, 0x7FC0, 0x7F80):          # 16384, NaN, +inf
        wp = w.copy()
        wp[V:] = pad
        assert impl(h, wp, 1.0, 9) == a


LINEAR_PINS = [pin_reduces_to_logits_oracle, pin_zero_weights, pin_torch_fp64, pin_padding_ignored]


@pytest.mark.parametrize("pin", LINEAR_PINS, ids=lambda f: f.__name__)
def test_linear_pin(pin):
    pin(oracle.linear_logp_row)


# ------------------------------------------------------ planted mistakes

def _mut_padding_included(h, w, tau, t):
    return oracle.linear_logp_row(h, w, tau, t, vreal=VPAD) if t < VPAD else math.nan


def _mut_no_tau(h, w, tau, t):
    return oracle.linear_logp_row(h, w, 1.0, t)


def _mut_bf16_logits(h, w, tau, t):
    """Mistake: the logits are rounded to bf16 before the softmax."""
    hf = oracle.bf16_bits_to_f32(h).astype(np.float64)
    wf = oracle.bf16_bits_to_f32(w[:V]).astype(np.float64)
    x = (wf @ hf).astype(np.float32)
    xb = (x.view(np.uint32) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16
    row = np.full(VPAD, 0xFF80, np.uint16)
    row[:V] = xb.astype(np.uint16)
    return oracle.logp_row(row, tau, 1.0, -1, t).full


@pytest.mark.parametrize("mutant", [_mut_padding_included, _mut_no_tau, _mut_bf16_logits],
                         ids=lambda f: f.__name__)
def test_planted_linear_mistake_is_caught(mutant):
    failed = []
    for pin in LINEAR_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"
