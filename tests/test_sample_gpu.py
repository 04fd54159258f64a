"""GPU: the sampler against the oracle's inverse-CDF draw.

The GPU draws filtered rows on exact fixed-point masses (2^-44 units of
exp((x - M)/tau), float32 exponent arguments and ex2.approx) and unfiltered
rows on float masses summed in a fixed order (chunks, 32-chunk words, a scan
over the words); the oracle draws on fp64 masses, so the two can pick
neighbouring tokens only when the draw U lies within 2e-6 of an edge of the
oracle's CDF; such rows are counted, everything else must match exactly.  The
sampled token's logprobs equal rlk_logp_pair's for that target bit for bit.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import rollout_consistent_vocab_gb300 as pkg
from rollout_consistent_vocab_gb300 import workloads as W

from _support import TOL, bits_of

pytestmark = pytest.mark.gpu
VR, VP = oracle.VREAL, oracle.VPAD
DEV = "cuda"
EDGE = 2e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rollout_consistent_vocab_gb300.build import build_library
    build_library()
    pkg.load_library()


def _t(a, dtype):
    return torch.as_tensor(np.asarray(a), dtype=dtype, device=DEV)


def _u32_tensor(u):
    return torch.as_tensor(np.asarray(u, dtype=np.uint32).view(np.int32), device=DEV)


def check_draws(bits, tau, p, k, u, tok, restr, full, sup):
    near = 0
    for i in range(bits.shape[0]):
        try:
            o = oracle.sample_row(bits[i], float(tau[i]), float(p[i]), int(k[i]), int(u[i]))
        except oracle.InvalidArgument:
            assert tok[i] == -1 and math.isnan(restr[i]) and sup[i] == -1, i
            continue
        if o.token == -1:
            assert tok[i] == -1 and math.isnan(full[i]) and sup[i] == -1, i
            continue
        if tok[i] != o.token:
            assert min(abs(o.u - o.lo_edge), abs(o.u - o.hi_edge)) <= EDGE, (i, tok[i], o.token)
            near += 1
        ref = oracle.logp_row(bits[i], float(tau[i]), float(p[i]), int(k[i]), int(tok[i]))
        assert math.isfinite(ref.restr), (i, "sampled token outside the support")
        assert abs(restr[i] - ref.restr) <= TOL and abs(full[i] - ref.full) <= TOL, i
        assert sup[i] == ref.support, (i, sup[i], ref.support)
    return near


def mixed(T, seed):
    rng = np.random.default_rng(seed)
    x, hot, n = W.hot_logits(T, 1, 300, seed=seed, device=DEV)
    tau = rng.choice([0.0, 0.5, 0.7, 1.0, 1.3, 2.0], T).astype(np.float32)
    p = rng.choice([0.5, 0.9, 0.95, 0.99, 0.9999, 1.0], T).astype(np.float32)
    k = rng.choice([-1, 1, 5, 50, 128, 1000, 3000], T).astype(np.int32)
    u = rng.integers(0, 2 ** 32, T, dtype=np.uint64).astype(np.uint32)
    return x, tau, p, k, u


def test_sampler_matches_oracle():
    x, tau, p, k, u = mixed(40, seed=41)
    # a NaN row, a rejected row, and two wide-support rows (nucleus crossing zero)
    x[36, 12345] = float("nan")
    tau[37] = -2.0
    xv = (0.02 * np.random.default_rng(41).standard_normal((2, VP))).astype(np.float32)
    xv[:, 5] = 3.0
    x[38:40] = torch.from_numpy(xv).to(DEV).to(torch.bfloat16)
    x[38:40, VR:] = float("-inf")
    tau[38:40], p[38:40], k[38:40] = 1.0, 0.9, -1
    bits = bits_of(x)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok, restr, full, sup = pkg.sample(x, _t(tau, torch.float32), _t(p, torch.float32),
                                       _t(k, torch.int32), uniform=_u32_tensor(u), err_count=err)
    torch.cuda.synchronize()
    assert err.item() == 1
    near = check_draws(bits, tau, p, k, u, tok.cpu().numpy(), restr.cpu().numpy(),
                       full.cpu().numpy(), sup.cpu().numpy())
    print("sampler rows near a CDF edge:", near)
    assert near <= 1


def test_sampler_logprobs_equal_the_pair_pass_bitwise():
    x, tau, p, k, u = mixed(64, seed=42)
    args = (_t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32))
    tok, restr, full, sup = pkg.sample(x, *args, uniform=_u32_tensor(u))
    f, r, s = pkg.logp_pair(x, tok.clamp(min=0), *args)
    torch.cuda.synchronize()
    ok = tok >= 0
    assert torch.equal(restr[ok].view(torch.int32), r[ok].view(torch.int32))
    assert torch.equal(full[ok].view(torch.int32), f[ok].view(torch.int32))
    assert torch.equal(sup, s)


def test_philox_draws_match_the_oracle_generator():
    x, tau, p, k, _ = mixed(24, seed=43)
    seed = 0x1234_5678_9ABC_DEF0
    ctr = np.arange(24, dtype=np.int64) * 7919 + (1 << 40)
    u = np.array([oracle.philox_uniform_bits(seed, int(c)) for c in ctr], dtype=np.uint32)
    args = (_t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32))
    a = pkg.sample(x, *args, seed=seed, counter=_t(ctr, torch.int64))
    b = pkg.sample(x, *args, uniform=_u32_tensor(u))
    torch.cuda.synchronize()
    for v, w in zip(a, b):
        assert torch.equal(v.view(torch.int32), w.view(torch.int32))


def test_sampler_is_batch_invariant():
    x, tau, p, k, _ = mixed(48, seed=44)
    ctr = _t(np.arange(48, dtype=np.int64) + 1000, torch.int64)
    args = (_t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32))
    t0, r0, f0, s0 = pkg.sample(x, *args, seed=99, counter=ctr)
    sub = torch.as_tensor([40, 3, 17, 17, 8, 29], device=DEV)
    big = torch.full((9, VP + 32), float("nan"), dtype=torch.bfloat16, device=DEV)
    big[3:, :VP] = x[sub]
    t1, r1, f1, s1 = pkg.sample(big[3:], *(a[sub].contiguous() for a in args), seed=99,
                                counter=ctr[sub].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(t1, t0[sub]) and torch.equal(s1, s0[sub])
    assert torch.equal(r1.view(torch.int32), r0[sub].view(torch.int32))


def test_stratified_frequencies():
    """One row drawn 2048 times with stratified words: each token of the support
    is drawn 2048 q_j times, up to one (two at the fixed-point CDF edges)."""
    x, _, _ = W.hot_logits(1, 40, 40, seed=45, device=DEV)
    n = 2048
    xs = x.expand(n, VP).contiguous()
    u = ((np.arange(n) + 0.5) * 2 ** 32 / n).astype(np.uint64).astype(np.uint32)
    tok, _, _, _ = pkg.sample(xs, 1.0, 0.95, 64, uniform=_u32_tensor(u))
    torch.cuda.synchronize()
    counts = np.bincount(tok.cpu().numpy(), minlength=VR)
    _, restr, S = oracle.row_logprobs_all(bits_of(x)[0], 1.0, 0.95, 64)
    assert counts[~S].sum() == 0
    assert np.all(np.abs(counts[S] - n * np.exp(restr[S])) <= 2.0)


def test_stratified_frequencies_unfiltered():
    """The same on an unfiltered row (top-p 1, top-k off: every real token in
    the support, drawn from the pair pass's word masses): each token drawn
    2048 q_j times, up to two."""
    x, _, _ = W.hot_logits(1, 40, 40, seed=46, device=DEV)
    n = 2048
    xs = x.expand(n, VP).contiguous()
    u = ((np.arange(n) + 0.5) * 2 ** 32 / n).astype(np.uint64).astype(np.uint32)
    tok, restr, full, sup = pkg.sample(xs, 1.0, 1.0, -1, uniform=_u32_tensor(u))
    torch.cuda.synchronize()
    assert (sup == VR).all() and torch.equal(restr.view(torch.int32), full.view(torch.int32))
    counts = np.bincount(tok.cpu().numpy(), minlength=VR)
    full_all, _, _ = oracle.row_logprobs_all(bits_of(x)[0], 1.0, 1.0, -1)
    assert counts.sum() == n
    assert np.all(np.abs(counts - n * np.exp(full_all)) <= 2.0)


def test_unfiltered_rows_match_the_oracle():
    """Unfiltered rows at several temperatures, drawn from the word masses:
    tokens against the oracle (edge rows counted), logprobs bit for bit."""
    x, _, _ = W.hot_logits(64, 1, 300, seed=47, device=DEV)
    rng = np.random.default_rng(47)
    tau = rng.choice([0.5, 0.7, 1.0, 1.3, 2.0], 64).astype(np.float32)
    p = np.ones(64, np.float32)
    k = np.full(64, -1, np.int32)
    u = rng.integers(0, 2 ** 32, 64, dtype=np.uint64).astype(np.uint32)
    tok, restr, full, sup = pkg.sample(x, _t(tau, torch.float32), 1.0, -1, uniform=_u32_tensor(u))
    torch.cuda.synchronize()
    near = check_draws(bits_of(x), tau, p, k, u, tok.cpu().numpy(), restr.cpu().numpy(),
                       full.cpu().numpy(), sup.cpu().numpy())
    print("unfiltered rows near a CDF edge:", near)
    assert near <= 1


def test_full_size_draws_are_in_support():
    """T = 8192 (the bench workload) with Philox counters: every token lies in
    its row's support and carries the pair pass's logprobs."""
    wl = W.workload_c2(device=DEV, with_ref=False)
    ctr = torch.arange(wl.T, device=DEV, dtype=torch.int64)
    tok, restr, full, sup = pkg.sample(wl.logits, 1.3, 0.99, 128, seed=2024, counter=ctr)
    f, r, s = pkg.logp_pair(wl.logits, tok, 1.3, 0.99, 128)
    torch.cuda.synchronize()
    assert (tok >= 0).all() and torch.isfinite(r).all()
    assert torch.equal(restr.view(torch.int32), r.view(torch.int32)) and torch.equal(sup, s)
    assert (sup <= 128 + 64).all()
    del wl
    torch.cuda.empty_cache()


def _sample_noalloc(x, tau, p, k, u):
    """The cluster draw for every row (rlk_sample_noalloc keeps no chunk bitmaps)."""
    import ctypes
    from rollout_consistent_vocab_gb300 import _binding as b
    lib = pkg.load_library()
    T = x.shape[0]
    a = b.make_args(x, None, tau, p, k)
    outs = (torch.empty(T, dtype=torch.int32, device=DEV), torch.empty(T, device=DEV),
            torch.empty(T, device=DEV), torch.empty(T, dtype=torch.int32, device=DEV))
    st = lib.rlk_sample_noalloc(ctypes.byref(a), 0, None, u.data_ptr(), outs[0].data_ptr(),
                                outs[1].data_ptr(), outs[2].data_ptr(), outs[3].data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert st == b.RLK_OK, lib.rlk_last_error()
    return outs


@pytest.mark.parametrize("case", ["bench_workload", "mixed"])
def test_bitmap_draw_equals_cluster_draw(case):
    """Rows whose support lies in the candidate window are drawn from the
    marked chunks alone; the result must equal the cluster draw's, which
    re-reads every shard, bit for bit (tokens, logprobs, supports)."""
    if case == "bench_workload":
        wl = W.workload_c2(device=DEV, with_ref=False)
        x, T = wl.logits, wl.T
        tau, p, k = _t([1.3] * T, torch.float32), _t([0.99] * T, torch.float32), _t([128] * T, torch.int32)
    else:
        x, tau_n, p_n, k_n, _ = mixed(2000, 71)
        T = x.shape[0]
        tau, p, k = _t(tau_n, torch.float32), _t(p_n, torch.float32), _t(k_n, torch.int32)
    rng = np.random.default_rng(72)
    u = _u32_tensor(rng.integers(0, 2 ** 32, T, dtype=np.uint64).astype(np.uint32))
    got = pkg.sample(x, tau, p, k, uniform=u)
    want = _sample_noalloc(x, tau, p, k, u)
    torch.cuda.synchronize()
    for g, w in zip(got, want):
        assert torch.equal(g.view(torch.int32), w.view(torch.int32))


def test_sampler_coarse_ties():
    """Logits quantised to 17 values: tie classes of thousands of tokens at
    every threshold, so the draw picks among equal-mass tokens (inverse CDF
    in column order) and supports take or drop whole classes.  Every row's
    token against the oracle's draw with the same random word."""
    T = 48
    rng = np.random.default_rng(47)
    g = torch.Generator(device=DEV).manual_seed(47)
    x = torch.full((T, VP), float("-inf"), device=DEV)
    x[:, :VR] = torch.clamp(torch.round(2.0 * torch.randn((T, VR), generator=g, device=DEV)) / 2.0, -4.0, 4.0)
    x = x.to(torch.bfloat16)
    tau = rng.choice([0.7, 1.0, 1.3], T).astype(np.float32)
    p = rng.choice([0.5, 0.9, 1.0], T).astype(np.float32)
    k = rng.choice([-1, 10, 1000], T).astype(np.int32)
    u = rng.integers(0, 2 ** 32, T, dtype=np.uint64).astype(np.uint32)
    bits = bits_of(x)
    tok, restr, full, sup = pkg.sample(x, _t(tau, torch.float32), _t(p, torch.float32),
                                       _t(k, torch.int32), uniform=_u32_tensor(u))
    torch.cuda.synchronize()
    near = check_draws(bits, tau, p, k, u, tok.cpu().numpy(), restr.cpu().numpy(),
                       full.cpu().numpy(), sup.cpu().numpy())
    assert near <= 1
