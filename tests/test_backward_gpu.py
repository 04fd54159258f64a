"""GPU: the backward pass (gradient of g_full * full + g_restr * restr with
respect to the logits) against the oracle, element by element.

Tolerance, per element: 2e-5 x (|g_full| |G_full_j| + |g_restr| |G_restr_j|)
with G the oracle's exact per-part gradients, plus 2e-6 (|g_full| + |g_restr|)
/ tau at the target column (where b - e_t a cancels).  The GPU's relative error
comes from float32 exponent arguments, ex2.approx and the float32 shard sums
(a few 1e-6); bf16 outputs add 2^-8 of the value.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import rollout_consistent_vocab_gb300 as pkg
from rollout_consistent_vocab_gb300 import workloads as W

from _support import bits_of, oracle_targets

pytestmark = pytest.mark.gpu
VR, VP = oracle.VREAL, oracle.VPAD
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rollout_consistent_vocab_gb300.build import build_library
    build_library()
    pkg.load_library()


def _t(a, dtype):
    return torch.as_tensor(np.asarray(a), dtype=dtype, device=DEV)


def check_grad_rows(bits, tau, p, k, t, gf, gr, got, bf16=False, rows=None):
    rows = range(bits.shape[0]) if rows is None else rows
    worst = 0.0
    for n, i in enumerate(rows):
        args = (float(tau[i]), float(p[i]), int(k[i]), int(t[i]))
        try:
            g1 = oracle.logp_grad_row(bits[n], *args, 1.0, 0.0)
            g2 = oracle.logp_grad_row(bits[n], *args, 0.0, 1.0)
        except oracle.InvalidArgument:
            assert np.all(np.isnan(got[n][:VR])) and np.all(got[n][VR:] == 0.0), i
            continue
        ref = gf[i] * g1 + gr[i] * g2
        if np.any(np.isnan(g1)):
            assert np.all(np.isnan(got[n][:VR])) and np.all(got[n][VR:] == 0.0), i
            continue
        tol = 2e-5 * (abs(gf[i]) * np.abs(g1) + abs(gr[i]) * np.abs(g2)) + 1e-30
        if args[0] > 0:
            tol[args[3]] += 2e-6 * (abs(gf[i]) + abs(gr[i])) / float(np.float32(args[0]))
        if bf16:
            # round to nearest: |bf16(v) - v| <= 2^-8 |v|, |v - ref| <= tol
            tol = tol * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ref)
        err = np.abs(got[n].astype(np.float64) - ref)
        bad = np.nonzero(err > tol)[0]
        assert len(bad) == 0, (i, args, bad[:5], got[n][bad[:5]], ref[bad[:5]])
        assert np.all(got[n][VR:] == 0.0)
        worst = max(worst, float(np.max(err / np.maximum(tol, 1e-300))))
    return worst


def mixed(T, seed):
    rng = np.random.default_rng(seed)
    x, hot, n = W.hot_logits(T, 1, 200, seed=seed, device=DEV)
    tau = rng.choice([0.0, 0.5, 0.7, 1.0, 1.3], T).astype(np.float32)
    p = rng.choice([0.5, 0.9, 0.95, 0.99, 1.0], T).astype(np.float32)
    k = rng.choice([-1, 1, 20, 128, 2000], T).astype(np.int32)
    bits = bits_of(x)
    forced = set(rng.choice(T, max(1, T // 5), replace=False).tolist())
    t = oracle_targets(bits, tau, p, k, rng, forced)
    gf = rng.standard_normal(T).astype(np.float32)
    gr = rng.standard_normal(T).astype(np.float32)
    return x, bits, tau, p, k, t, gf, gr


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_backward_matches_oracle(dtype):
    x, bits, tau, p, k, t, gf, gr = mixed(14, seed=31)
    # extra rows: a NaN row and a rejected row
    x = torch.cat([x, x[:2]])
    x[14, 777] = float("nan")
    tau = np.append(tau, [0.7, -1.0]).astype(np.float32)
    p, k = np.append(p, [0.9, 0.9]).astype(np.float32), np.append(k, [-1, -1]).astype(np.int32)
    t, gf, gr = np.append(t, [5, 5]), np.append(gf, [1, 1]).astype(np.float32), np.append(gr, [1, 1]).astype(np.float32)
    bits = bits_of(x)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    g = pkg.logp_backward(x, _t(t, torch.int32), _t(tau, torch.float32), _t(p, torch.float32),
                          _t(k, torch.int32), grad_full=_t(gf, torch.float32),
                          grad_restr=_t(gr, torch.float32), dtype=dtype, err_count=err)
    torch.cuda.synchronize()
    assert err.item() == 1
    got = g.float().cpu().numpy()
    worst = check_grad_rows(bits, tau, p, k, t, gf, gr, got, bf16=dtype == torch.bfloat16)
    for i in np.nonzero(tau == 0.0)[0]:
        assert np.all(got[i] == 0.0)
    print("backward", dtype, "worst err/tol", worst)


def test_backward_full_only_and_restricted_only():
    x, bits, tau, p, k, t, gf, gr = mixed(8, seed=32)
    tt, ta, pa, ka = _t(t, torch.int32), _t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32)
    g_full = pkg.logp_backward(x, tt, ta, grad_full=_t(gf, torch.float32), dtype=torch.float32)
    g_restr = pkg.logp_backward(x, tt, ta, pa, ka, grad_restr=_t(gr, torch.float32), dtype=torch.float32)
    torch.cuda.synchronize()
    zeros = np.zeros_like(gf)
    ones_p, none_k = np.ones_like(p), -np.ones_like(k)
    check_grad_rows(bits, tau, ones_p, none_k, t, gf, zeros, g_full.cpu().numpy())
    check_grad_rows(bits, tau, p, k, t, zeros, gr, g_restr.cpu().numpy())


def test_backward_forward_outputs_and_invariance():
    """The forward outputs of the backward pass equal logp_pair bit for bit, and
    a row's gradient bits do not depend on the batch around it or its buffer."""
    x, bits, tau, p, k, t, gf, gr = mixed(40, seed=33)
    args = (_t(t, torch.int32), _t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32))
    f, r, s = torch.empty(40, device=DEV), torch.empty(40, device=DEV), torch.empty(40, dtype=torch.int32, device=DEV)
    g = pkg.logp_backward(x, *args, grad_full=_t(gf, torch.float32), grad_restr=_t(gr, torch.float32),
                          out_full=f, out_restr=r, out_support=s)
    f0, r0, s0 = pkg.logp_pair(x, *args)
    sub = slice(3, 11)
    big = torch.full((12, VP + 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    big[4:, :VP] = x[sub]
    gsub = torch.full((8, VP + 16), 7.0, dtype=torch.bfloat16, device=DEV)
    pkg.logp_backward(big[4:], *(a[sub] for a in args), grad_full=_t(gf[sub], torch.float32),
                      grad_restr=_t(gr[sub], torch.float32), out=gsub)
    torch.cuda.synchronize()
    for u, v in ((f, f0), (r, r0)):
        assert torch.equal(u.view(torch.int32), v.view(torch.int32))
    assert torch.equal(s, s0)
    assert torch.equal(gsub[:, :VP].view(torch.int16), g[sub].view(torch.int16))
    assert (gsub[:, VP:] == 7.0).all()      # nothing written past the row


def test_backward_wide_support_rows():
    """Rows whose support reaches below the window: the leader's shard copy is
    reused as scratch by the fallback selection and its gradient is written
    from global memory instead."""
    rng = np.random.default_rng(34)
    T = 6
    xv = (0.02 * rng.standard_normal((T, VP))).astype(np.float32)
    xv[:, 5] = 3.0
    bits = (xv.view(np.uint32) >> 16).astype(np.uint16)
    bits[:, VR:] = 0xFF80
    tau = np.array([1.0, 1.0, 0.5, 1.0, 2.0, 1.0], np.float32)
    p = np.array([0.9, 0.5, 0.99, 1.0, 0.7, 0.99], np.float32)
    k = np.array([-1, -1, -1, 100000, 70000, 3000], np.int32)
    t = oracle_targets(bits, tau, p, k, rng, {1})
    gf = rng.standard_normal(T).astype(np.float32)
    gr = rng.standard_normal(T).astype(np.float32)
    x = torch.from_numpy(bits.view(np.int16).copy()).to(DEV).view(torch.bfloat16)
    g = pkg.logp_backward(x, _t(t, torch.int32), _t(tau, torch.float32), _t(p, torch.float32),
                          _t(k, torch.int32), grad_full=_t(gf, torch.float32),
                          grad_restr=_t(gr, torch.float32), dtype=torch.float32)
    torch.cuda.synchronize()
    check_grad_rows(bits, tau, p, k, t, gf, gr, g.cpu().numpy())


def _okey(b):
    b = int(b)
    if b == 0x8000:
        return 0x8000
    return (~b & 0xFFFF) if b & 0x8000 else (b | 0x8000)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_saved_backward_equals_single_pass(dtype):
    """pair_save + backward_saved gives the single-pass backward's bits,
    on mixed rows, NaN rows, rejected rows and wide-support rows."""
    x, bits, tau, p, k, t, gf, gr = mixed(24, seed=37)
    x[20, 5000] = float("nan")
    tau[21] = -1.0
    xv = (0.02 * np.random.default_rng(37).standard_normal((2, VP))).astype(np.float32)
    xv[:, 5] = 3.0
    x[22:24] = torch.from_numpy(xv).to(DEV).to(torch.bfloat16)
    x[22:24, VR:] = float("-inf")
    p[22:24], k[22:24], tau[22:24] = 0.9, -1, 1.0
    args = (_t(t, torch.int32), _t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32))
    gfa, gra = _t(gf, torch.float32), _t(gr, torch.float32)
    g1 = pkg.logp_backward(x, *args, grad_full=gfa, grad_restr=gra, dtype=dtype)
    f, r, s, stats = pkg.logp_pair_save(x, *args)
    g2 = pkg.logp_backward_saved(x, args[0], stats, args[1], grad_full=gfa, grad_restr=gra, dtype=dtype)
    f0, r0, s0 = pkg.logp_pair(x, *args)
    torch.cuda.synchronize()
    iv = torch.int32 if dtype == torch.float32 else torch.int16
    assert torch.equal(g1.view(iv), g2.view(iv))
    assert torch.equal(f.view(torch.int32), f0.view(torch.int32)) and torch.equal(s, s0)
    assert torch.equal(r.view(torch.int32), r0.view(torch.int32))


def test_saved_record_matches_the_oracle():
    """The per-row record: M exact, 1/Z and 1/Z_S within 1e-5 relative of the
    oracle's sums, the support's lowest key exact, 0 when t is outside S."""
    x, bits, tau, p, k, t, gf, gr = mixed(16, seed=38)
    args = (_t(t, torch.int32), _t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32))
    _, restr, sup, stats = pkg.logp_pair_save(x, *args)
    torch.cuda.synchronize()
    st = stats.cpu().numpy()
    mk = stats.view(torch.int32)[:, 3].cpu().numpy()
    rv = restr.cpu().numpy()
    for i in range(16):
        xs = oracle.bf16_bits_to_f32(bits[i][:VR]).astype(np.float64)
        M = xs.max()
        assert st[i, 0] == M
        if tau[i] == 0.0:
            assert st[i, 1] == 0.0
            continue
        s = oracle.scaled_logits(bits[i], float(tau[i]))
        w = np.exp(s - s.max())
        assert abs(st[i, 1] * math.fsum(w) - 1.0) < 1e-5, i
        sk = oracle.top_k_mask(s, int(k[i]))
        S = oracle.top_p_mask(s, sk, float(p[i]))[0] if p[i] < 1.0 else sk
        if rv[i] == -math.inf:
            assert st[i, 2] == 0.0
        else:
            assert abs(st[i, 2] * math.fsum(w[S]) - 1.0) < 1e-5, i
        want_key = min(_okey(b) for b in bits[i][:VR][S]) if S.sum() < VR else 0
        if S.sum() < VR:
            assert mk[i] == want_key, (i, mk[i], want_key)


def test_autograd_wrapper():
    x, bits, tau, p, k, t, gf, gr = mixed(6, seed=35)
    tau = np.maximum(tau, 0.5).astype(np.float32)
    xs = x.clone().requires_grad_(True)
    args = (_t(t, torch.int32), _t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32))
    full, restr = pkg.logp_autograd(xs, *args)
    gfa, gra = _t(gf, torch.float32), _t(gr, torch.float32)
    restr_finite = torch.where(torch.isinf(restr), torch.zeros_like(restr), restr)
    loss = (full * gfa).sum() + (restr_finite * gra).sum()
    (gx,) = torch.autograd.grad(loss, xs)
    want = pkg.logp_backward(x, *args, grad_full=gfa, grad_restr=gra * torch.isfinite(restr))
    torch.cuda.synchronize()
    assert torch.equal(gx.view(torch.int16), want.view(torch.int16))


def test_backward_full_size_sampled_rows():
    """T = 8192 (the bench workload): every row's gradient sums to ~0 (softmax
    gradients), and sampled rows match the oracle."""
    wl = W.workload_c2(device=DEV, with_ref=False)
    T = wl.T
    tg = W.structural_targets(T, wl.hot, wl.hot_n, seed=2, device=DEV)
    g_full = torch.randn(T, generator=torch.Generator(device=DEV).manual_seed(5), device=DEV)
    g_restr = torch.randn(T, generator=torch.Generator(device=DEV).manual_seed(6), device=DEV)
    g = pkg.logp_backward(wl.logits, tg, 1.3, 0.99, 128, grad_full=g_full, grad_restr=g_restr,
                          dtype=torch.float32)
    _, _, _, stats = pkg.logp_pair_save(wl.logits, tg, 1.3, 0.99, 128)
    g2 = pkg.logp_backward_saved(wl.logits, tg, stats, 1.3, grad_full=g_full, grad_restr=g_restr,
                                 dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(g.view(torch.int32), g2.view(torch.int32))
    del g2
    sums = g.double().sum(1)
    scale = (g_full.abs() + g_restr.abs()).double() / 1.3
    assert (sums.abs() <= 1e-5 * scale + 1e-12).all(), sums.abs().max().item()
    rng = np.random.default_rng(36)
    rows = np.sort(rng.choice(T, 6, replace=False))
    ridx = torch.as_tensor(rows, device=DEV)
    bits = bits_of(wl.logits[ridx])
    ones = np.ones(T)
    check_grad_rows(bits, 1.3 * ones, 0.99 * ones, 128 * ones, tg.cpu().numpy(),
                    g_full.cpu().numpy(), g_restr.cpu().numpy(), g[ridx].cpu().numpy(), rows=rows)
    del g, wl
    torch.cuda.empty_cache()


def test_backward_coarse_ties():
    """Logits quantised to 17 values: the support takes or drops tie classes
    of thousands of tokens, so each class's gradient is either all inside
    (a_in) or all outside (a_out).  Both backward forms against the oracle,
    element by element."""
    T = 10
    rng = np.random.default_rng(37)
    g = torch.Generator(device=DEV).manual_seed(37)
    x = torch.full((T, VP), float("-inf"), device=DEV)
    x[:, :VR] = torch.clamp(torch.round(2.0 * torch.randn((T, VR), generator=g, device=DEV)) / 2.0, -4.0, 4.0)
    x = x.to(torch.bfloat16)
    tau = rng.choice([0.7, 1.3], T).astype(np.float32)
    p = rng.choice([0.5, 0.9, 1.0], T).astype(np.float32)
    k = rng.choice([-1, 10, 1000], T).astype(np.int32)
    bits = bits_of(x)
    t = oracle_targets(bits, tau, p, k, rng, set(rng.choice(T, 2, replace=False).tolist()))
    gf = rng.standard_normal(T).astype(np.float32)
    gr = rng.standard_normal(T).astype(np.float32)
    args = (_t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32))
    single = pkg.logp_backward(x, _t(t, torch.int32), *args, grad_full=_t(gf, torch.float32),
                               grad_restr=_t(gr, torch.float32), dtype=torch.float32)
    _, _, _, stats = pkg.logp_pair_save(x, _t(t, torch.int32), *args)
    saved = torch.empty((T, VP), dtype=torch.float32, device=DEV)
    pkg.logp_backward_saved(x, _t(t, torch.int32), stats, _t(tau, torch.float32),
                            grad_full=_t(gf, torch.float32), grad_restr=_t(gr, torch.float32),
                            out=saved)
    torch.cuda.synchronize()
    for got in (single, saved):
        check_grad_rows(bits, tau, p, k, t, gf, gr, got.cpu().numpy())
