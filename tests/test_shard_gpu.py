"""GPU: the vocabulary-sharded entry points (per-shard summaries, per-shard
candidate counts, merge) against the fused kernel and the oracle.

The fused kernel and the sharded form run the same per-shard passes and the
same fixed-order merge, so full logprobs must agree bit for bit, and so must
the restricted logprob and support of every row: rows whose support reaches
below the first 1024-key window are carried through lower windows by the
resumable merge (one merge round alone reports them with support -2).  The
shard summaries themselves are checked against the oracle's fp64 summaries.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import rollout_consistent_vocab_gb300 as pkg
from rollout_consistent_vocab_gb300 import workloads as W

from _support import bits_of

pytestmark = pytest.mark.gpu
VR, VP, SW, NS = oracle.VREAL, oracle.VPAD, oracle.SHARD_W, oracle.NSHARD
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rollout_consistent_vocab_gb300.build import build_library
    build_library()
    pkg.load_library()


def split(x: torch.Tensor):
    """The 8 shard buffers a tensor-parallel rank would hold: [T, 19072] each."""
    return [x[:, r * SW:(r + 1) * SW].contiguous() for r in range(NS)]


def bits32(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int32).cpu().numpy()


def _t(a, dtype):
    return torch.as_tensor(np.asarray(a), dtype=dtype, device=DEV)


def mixed_rows(T: int, seed: int):
    """Hot rows with per-row tau/p/k spanning greedy, top-k only, top-p only,
    both, disabled, and k above the pooled-witness range (k > 1024)."""
    rng = np.random.default_rng(seed)
    x, hot, n = W.hot_logits(T, 1, 300, seed=seed, device=DEV)
    t = W.structural_targets(T, hot, n, seed=seed, device=DEV)
    tau = rng.choice([0.0, 0.5, 0.7, 1.0, 1.3, 2.0], T).astype(np.float32)
    p = rng.choice([0.5, 0.9, 0.95, 0.99, 0.9999, 1.0], T).astype(np.float32)
    k = rng.choice([-1, 1, 5, 50, 128, 1000, 1024, 1025, 3000], T).astype(np.int32)
    return x, t, _t(tau, torch.float32), _t(p, torch.float32), _t(k, torch.int32)


def compare(x, t, tau, p, k, err=None, err_sharded=None):
    """Fused pass against the sharded form: bit for bit on every row (rows
    beyond the first window resolved over lower windows).  Also returns the
    supports of a single merge round, where such rows report -2."""
    f0, r0, s0 = pkg.logp_pair(x, t, tau, p, k, err_count=err)
    f1, r1, s1 = pkg.logp_sharded(split(x), t, tau, p, k, err_count=err_sharded)
    # phase 2 reading whole shards instead of the chunks phase 1 marked: the same bits
    f2, r2, s2 = pkg.logp_sharded(split(x), t, tau, p, k, chunk_maxima=False)
    # one merge round: rows outside the first window stay at support -2
    f3, r3, s3 = pkg.logp_sharded(split(x), t, tau, p, k, resolve=False)
    torch.cuda.synchronize()
    for u, v in ((f1, f2), (r1, r2), (s1, s2)):
        assert torch.equal(u.view(torch.int32), v.view(torch.int32))
    for fx in (f1, f3):
        f0b, fxb = bits32(f0), bits32(fx)
        assert (f0b == fxb).all(), np.nonzero(f0b != fxb)[0][:10]
    s0n, s1n, s3n = s0.cpu().numpy(), s1.cpu().numpy(), s3.cpu().numpy()
    r0b, r1b, r3b = bits32(r0), bits32(r1), bits32(r3)
    bad = np.nonzero((r0b != r1b) | (s0n != s1n))[0]
    assert len(bad) == 0, (bad[:10], s0n[bad[:10]], s1n[bad[:10]])
    ok = s3n != -2
    assert ((r3b == r0b) | ~ok).all() and ((s3n == s0n) | ~ok).all()
    # rows outside the first window: NaN restricted after one round, a real support in the fused kernel
    wide = np.nonzero(~ok)[0]
    assert np.isnan(r3.cpu().numpy()[wide]).all()
    assert (s0n[wide] > 0).all()
    return s0n, s3n


def test_sharded_matches_fused_mixed_parameters():
    x, t, tau, p, k = mixed_rows(300, seed=21)
    s0, s1 = compare(x, t, tau, p, k)
    # only deep supports (p = 0.9999, k = 3000: far more tokens than the largest
    # hot set of 300) may reach below the window
    wide = s1 == -2
    assert wide.sum() <= len(s1) // 20 and (s0[wide] > 300).all(), s0[wide]


def test_sharded_full_only_matches_logp_full():
    x, t, tau, p, k = mixed_rows(64, seed=22)
    f0 = pkg.logp_full(x, t, tau)
    (f1,) = pkg.logp_sharded(split(x), t, tau, restricted=False)
    torch.cuda.synchronize()
    assert (bits32(f0) == bits32(f1)).all()


def test_sharded_nonfinite_and_invalid_rows():
    base, hot, n = W.hot_logits(12, 1, 32, seed=23, device=DEV)
    x = base.clone()
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    x[0, 3 * SW:4 * SW] = nan                               # one whole shard NaN
    for i in range(19):                                      # every chunk one thread owns
        c = 2 * SW + (5 + 128 * i) * 8
        if c + 8 <= 3 * SW:
            x[1, c:c + 8] = nan
    x[2, 1000] = float("inf")
    x[3, 5 * SW:6 * SW] = float("-inf")                      # a shard with nothing in it
    x[4, VR - 1] = nan                                       # last real column
    x[5, VR:] = nan                                          # padding only: ignored
    t = W.structural_targets(12, hot, n, seed=23, device=DEV)
    tau = _t([0.7, 0.7, 0.7, 1.0, 0.0, 0.7, -1.0, 0.7, 0.7, 0.7, 0.7, 0.7], torch.float32)
    p = _t([0.9, 0.9, 0.9, 0.95, 1.0, 0.9, 0.9, 0.0, 0.9, 0.9, 0.9, 0.9], torch.float32)
    k = _t([50, -1, 50, -1, -1, 128, -1, -1, 0, -1, 50, 1], torch.int32)
    t[9] = VR
    err0 = torch.zeros(1, dtype=torch.int32, device=DEV)
    err1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    compare(x, t, tau, p, k, err0, err1)
    assert err0.item() == 4 and err1.item() == 4
    f, r, s = pkg.logp_pair(x, t, tau, p, k)
    torch.cuda.synchronize()
    for i in (0, 1, 2, 4):
        assert math.isnan(f[i].item()) and s[i].item() == -1, i
    assert not math.isnan(f[3].item()) and not math.isnan(f[5].item())


def test_sharded_spread_rows_and_wide_supports():
    """Spread rows (N(0,3^2), tau 0.7, p 0.95) keep their nucleus inside the
    window; rows centred on 0 with a small spread, whose nucleus crosses zero
    (many binades below the maximum), need lower windows: one merge round
    reports them with support -2, the resumable rounds resolve them to the
    fused kernel's bits (top-p alone, top-k alone, and top-k reaching below
    the window followed by top-p from the top window again)."""
    wl = W.workload_c0(device=DEV, T=32)
    t = W.structural_targets(32, None, None, seed=24, device=DEV)
    s0, s1 = compare(wl.logits, t, 0.7, 0.95, -1)
    assert (s1 != -2).all()
    g = torch.Generator(device=DEV).manual_seed(24)
    x = (0.02 * torch.randn((6, VP), generator=g, device=DEV)).to(torch.bfloat16)
    x[:, 5] = 3.0
    x[:, VR:] = float("-inf")
    t = torch.full((6,), 5, dtype=torch.int32, device=DEV)
    p = _t([0.9, 0.5, 0.99, 1.0, 0.7, 0.99], torch.float32)
    k = _t([-1, -1, -1, 100000, 70000, 3000], torch.int32)
    s0, s1 = compare(x, t, 1.0, p, k)
    assert (s1 == -2).sum() >= 4


def test_presummed_counts_and_stride():
    """count_shards = 1 (counts already summed across shards) and shard
    buffers inside wider rows give the same results."""
    x, t, tau, p, k = mixed_rows(40, seed=25)
    shards = split(x)
    T = x.shape[0]
    maxes = torch.empty((NS, T), dtype=torch.float32, device=DEV)
    sumexps = torch.empty_like(maxes)
    aux = torch.empty((NS, T), dtype=torch.int32, device=DEV)
    xt = torch.empty((T,), dtype=torch.float32, device=DEV)
    for r, sh in enumerate(shards):
        wide = torch.full((T, SW + 24), float("nan"), dtype=torch.bfloat16, device=DEV)
        wide[:, :SW] = sh
        pkg.shard_summary(wide, r, t, tau, p, k, out_max=maxes[r], out_sumexp=sumexps[r],
                          out_aux=aux[r], out_target_logit=xt)
    counts = torch.empty((NS, T, 1024), dtype=torch.int32, device=DEV)
    for r, sh in enumerate(shards):
        pkg.shard_counts(sh, r, t, maxes, sumexps, aux, tau, p, k, out_counts=counts[r])
    summed = counts.sum(0, keepdim=True, dtype=torch.int32)
    a = pkg.logp_merge(maxes, sumexps, aux, xt, t, tau, p, k, counts=counts)
    b = pkg.logp_merge(maxes, sumexps, aux, xt, t, tau, p, k, counts=summed)
    c = pkg.logp_pair(x, t, tau, p, k)
    torch.cuda.synchronize()
    for u, v, w in zip(a, b, c):
        assert (bits32(u) == bits32(v)).all() and (bits32(u) == bits32(w)).all()


def test_shard_summaries_match_the_oracle():
    """(max, sum-exp) of every shard against the oracle's fp64 summaries."""
    x, hot, n = W.hot_logits(6, 1, 64, seed=26, device=DEV)
    t = W.structural_targets(6, hot, n, seed=26, device=DEV)
    taus = [0.7, 1.0, 1.3, 2.0, 0.5, 1.0]
    tau = _t(taus, torch.float32)
    T = 6
    maxes = torch.empty((NS, T), dtype=torch.float32, device=DEV)
    sumexps = torch.empty_like(maxes)
    aux = torch.empty((NS, T), dtype=torch.int32, device=DEV)
    xt = torch.empty((T,), dtype=torch.float32, device=DEV)
    for r, sh in enumerate(split(x)):
        pkg.shard_summary(sh, r, t, tau, 1.0, -1, out_max=maxes[r], out_sumexp=sumexps[r],
                          out_aux=aux[r], out_target_logit=xt)
    torch.cuda.synchronize()
    bits = bits_of(x)
    m, l = maxes.cpu().numpy(), sumexps.cpu().numpy()
    for i in range(T):
        om, ol = oracle.shard_summaries(bits[i], taus[i])
        for r in range(NS):
            assert float(np.float32(m[r, i]) / np.float32(taus[i])) == om[r]
            assert abs(l[r, i] - ol[r]) <= 2e-5 * ol[r], (i, r, l[r, i], ol[r])
        assert xt[i].item() == float(oracle.bf16_bits_to_f32(bits[i][t[i].item():t[i].item() + 1])[0])


def test_sharded_resolves_every_row_of_deep_top_p_workloads():
    """Top-p-only rows at temperature 1.3 and p 0.99 (supports of thousands of
    tokens), the fused kernel's wide-support rows, and k beyond 1024 with top-p:
    through the sharded entry points every row resolves, bit for bit equal to
    the fused pass, and no row keeps support -2."""
    x, hot, n = W.hot_logits(48, 1, 512, seed=27, device=DEV)
    t = W.structural_targets(48, hot, n, seed=27, device=DEV)
    s0, s3 = compare(x, t, 1.3, 0.99, -1)
    assert (s0 > 1000).sum() >= 10
    rng = np.random.default_rng(28)
    xw = (0.02 * rng.standard_normal((8, VP))).astype(np.float32)
    xw[:, 5] = 3.0
    xw = torch.as_tensor(xw, device=DEV).to(torch.bfloat16)
    xw[:, VR:] = float("-inf")
    tw = _t([5, 9, 5, 77, 5, 1000, 5, 151935], torch.int32)
    tau = _t([1.0, 1.0, 0.5, 1.0, 2.0, 1.0, 1.0, 1.0], torch.float32)
    p = _t([0.9, 0.5, 0.99, 1.0, 0.7, 0.99, 0.3, 0.999], torch.float32)
    k = _t([-1, -1, -1, 100000, 70000, 3000, 120000, 20000], torch.int32)
    s0, s3 = compare(xw, tw, tau, p, k)
    assert (s3 == -2).sum() >= 5


def test_sharded_coarse_ties_bitwise():
    """Logits quantised to 17 values (tie classes of thousands of tokens at
    every threshold, supports reaching below the first window): the sharded
    form bit for bit against the fused pass on every row."""
    T = 64
    rng = np.random.default_rng(43)
    g = torch.Generator(device=DEV).manual_seed(43)
    x = torch.full((T, VP), float("-inf"), device=DEV)
    x[:, :VR] = torch.clamp(torch.round(2.0 * torch.randn((T, VR), generator=g, device=DEV)) / 2.0, -4.0, 4.0)
    x = x.to(torch.bfloat16)
    tau = torch.as_tensor(rng.choice([0.7, 1.0, 1.3], T).astype(np.float32), device=DEV)
    p = torch.as_tensor(rng.choice([0.5, 0.9, 0.99, 1.0], T).astype(np.float32), device=DEV)
    k = torch.as_tensor(rng.choice([-1, 1, 10, 1000, 50000], T).astype(np.int32), device=DEV)
    t = torch.as_tensor(rng.integers(0, VR, T).astype(np.int32), device=DEV)
    compare(x, t, tau, p, k)
