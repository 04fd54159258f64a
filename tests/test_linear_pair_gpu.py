"""GPU: full and restricted logprob straight from the LM head
(rlk_linear_logp_pair) against the oracle's exact logits
(oracle.linear_logp_pair_rows).

Tolerance, from the arithmetic: the tensor cores accumulate each logit in
fp32 over K/16 steps, each rounding at most 2^-24 of the running sum, which
is bounded by S = max_j sum_k |h_k W_jk|; as a random walk that is
delta = 4 sqrt(K/16) 2^-24 S with a 4-sigma margin, so each scaled logit
moves by eps = delta / tau.  Both logprobs then move by at most 2 eps, plus
2e-5 for the exponentials and the logarithm (the bound of the logits path).

Supports.  The GPU selects exactly on its own fp32 logits, the oracle on the
exact ones, so a decision can differ where eps can flip it.  A GPU support of
size n' is accepted when it is the outcome of some perturbation of the exact
scaled logits by at most eps each:
  * top-k: every token the GPU keeps beyond the exact k-th largest value, or
    drops above it, lies within 2 eps of that value;
  * top-p: with the tokens in exact descending order, A_j the mass strictly
    above position j and Z the mass of the top-k set, such a perturbation
    moves every ratio A_j / Z by a factor within exp(+-2 eps) (plus 1e-6 for
    the fixed-point masses and the float normaliser): the last kept position
    must satisfy A / Z < p exp(2 eps) + 1e-6, the first dropped one
    A / Z >= p exp(-2 eps) - 1e-6.
Such rows are counted (support_differs) and scored on the GPU's support size
(the top n' tokens in exact order); where the target itself lies within 2 eps
of that support's edge its restricted value is not scored (target_at_edge).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import rollout_consistent_vocab_gb300 as pkg
from _oracle_check import record

pytestmark = pytest.mark.gpu
DEV = "cuda"
VR, VP = oracle.VREAL, oracle.VPAD


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rollout_consistent_vocab_gb300.build import build_library
    build_library()
    pkg.load_library()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _case(T, H, seed, hot=True, scale=4.0):
    """hidden [T, H], weight [VP, H]: logits about scale * N(0, 1); with `hot`,
    16 topic directions of 64 tokens each add +12 to a row's tokens of every
    topic it has active (each with probability 0.15)."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    h = torch.randn((T, H), generator=g, device=DEV)
    w = scale / H ** 0.5 * torch.randn((VP, H), generator=g, device=DEV)
    if hot:
        nt = 16
        toks = torch.randint(0, VR, (nt, 64), generator=g, device=DEV)
        for d in range(nt):
            w[toks[d], d] = 4.0
        act = torch.rand((T, nt), generator=g, device=DEV) < 0.15
        h[:, :nt] = torch.where(act, 3.0, 0.0)
    return h.to(torch.bfloat16), w.to(torch.bfloat16)


def _exact_logits(hb, wb):
    """x = W h in fp64 on the host (bf16 products are exact in fp64)."""
    hf = torch.from_numpy(oracle.bf16_bits_to_f32(hb).astype(np.float64))
    wf = torch.from_numpy(oracle.bf16_bits_to_f32(wb[:VR]).astype(np.float64))
    return (hf @ wf.T).numpy(), (hf.abs() @ wf.abs().T).max(dim=1).values.numpy()


def _targets(x, seed):
    """Half the rows: a token among the row's 32 largest logits; the rest uniform."""
    rng = np.random.default_rng(seed)
    T = x.shape[0]
    t = rng.integers(0, VR, T)
    top = np.argsort(-x, axis=1, kind="stable")[:, :32]
    pick = rng.random(T) < 0.5
    t[pick] = top[pick, rng.integers(0, 32, T)[pick]]
    return t.astype(np.int32)


def _delta(S, H):
    return 4 * math.sqrt(H / 16) * 2.0 ** -24 * S


class PairStats:
    def __init__(self):
        self.rows = self.support_differs = self.target_at_edge = 0
        self.max_full = self.max_restr = 0.0

    def as_dict(self):
        return dict(rows=self.rows, near_rows=self.support_differs, near_tokens=self.support_differs,
                    support_differs=self.support_differs, target_at_edge=self.target_at_edge,
                    max_full=self.max_full, max_restr=self.max_restr, max_kl=0.0)


def _plausible(s_desc, k, p, n_gpu, eps):
    """Whether a support of n_gpu tokens is the exact outcome for some
    perturbation of the scaled logits by at most eps (rule in the module
    docstring); s_desc: exact scaled logits, descending."""
    n = s_desc.shape[0]
    k_on = not (k == -1 or k >= n)
    if k_on:
        vk = s_desc[k - 1]
        nk_lo = max(k, int(np.count_nonzero(s_desc >= vk + 2 * eps)))
        nk_hi = int(np.count_nonzero(s_desc >= vk - 2 * eps))
    else:
        nk_lo = nk_hi = n
    if p >= 1.0:
        return nk_lo <= n_gpu <= nk_hi
    if not (1 <= n_gpu <= nk_hi):
        return False
    with np.errstate(under="ignore"):
        e = np.exp(s_desc - s_desc[0])
    above = np.concatenate(([0.0], np.cumsum(e)[:-1]))
    lo_f, hi_f = math.exp(-2 * eps), math.exp(2 * eps)
    for nk in range(nk_lo, min(nk_hi, nk_lo + 64) + 1):
        if n_gpu > nk:
            continue
        z = math.fsum(e[:nk])
        keep_ok = above[n_gpu - 1] / z < p * hi_f + 1e-6
        drop_ok = n_gpu == nk or above[n_gpu] / z >= p * lo_f - 1e-6
        if keep_ok and drop_ok:
            return True
    return False


def check_pair(name, hb, wb, x, S, H, taus, ps, ks, tg, full, restr, sup, stats=None):
    """Every row against the oracle, with the derived tolerance and support rule."""
    T = hb.shape[0]
    taus, ps, ks = (np.broadcast_to(np.asarray(v), (T,)) for v in (taus, ps, ks))
    o_full, o_restr, o_sup = oracle.linear_logp_pair_rows(hb, wb, taus, ps, ks, tg)
    st = stats if stats is not None else PairStats()
    for i in range(T):
        tau, p, k = float(taus[i]), float(ps[i]), int(ks[i])
        eps = _delta(S[i], H) / tau
        tol = 2e-5 + 2 * eps
        ctx = f"row {i} tau={tau} p={p} k={k} t={tg[i]}"
        assert abs(full[i] - o_full[i]) <= tol, (full[i], o_full[i], tol, ctx)
        st.max_full = max(st.max_full, abs(full[i] - o_full[i]))
        st.rows += 1
        want = o_restr[i]
        if sup[i] != o_sup[i]:
            s = x[i] / float(np.float32(tau))
            order = np.argsort(-s, kind="stable")
            sd = s[order]
            assert _plausible(sd, k, p, int(sup[i]), eps), (int(sup[i]), int(o_sup[i]), ctx)
            st.support_differs += 1
            n = int(sup[i])
            st_t = s[tg[i]]
            edge = abs(st_t - sd[n - 1]) <= 2 * eps or (n < VR and abs(st_t - sd[n]) <= 2 * eps)
            if edge:
                st.target_at_edge += 1
                continue
            m = sd[0]
            with np.errstate(under="ignore"):
                zs = math.fsum(np.exp(sd[:n] - m))
            want = (st_t - m) - math.log(zs) if st_t >= sd[n - 1] else -math.inf
        if math.isinf(want):
            assert restr[i] == want, (restr[i], want, ctx)
        else:
            assert abs(restr[i] - want) <= tol, (restr[i], want, tol, ctx)
            st.max_restr = max(st.max_restr, abs(restr[i] - want))
    if stats is None:
        record(name, st.as_dict())
        print(name, st.as_dict())
    return st


def _run(T, H, seed, taus, ps, ks, hot=True, scale=4.0):
    h, w = _case(T, H, seed, hot=hot, scale=scale)
    hb, wb = _bits(h), _bits(w)
    x, S = _exact_logits(hb, wb)
    tg = _targets(x, seed)
    dev = lambda v, dt: torch.as_tensor(v, dtype=dt, device=DEV) if np.ndim(v) else v
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    full, restr, sup = pkg.linear_logp_pair(h, w, torch.as_tensor(tg, device=DEV), dev(taus, torch.float32),
                                            dev(ps, torch.float32), dev(ks, torch.int32), err_count=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return (h, w, hb, wb, x, S, tg, full.cpu().numpy(), restr.cpu().numpy(), sup.cpu().numpy())


CONFIGS = {
    # name: (tau, top_p, top_k)
    "top_p_only_t0.7_p0.95": (0.7, 0.95, -1),           # the microbatch parameters
    "top_k_top_p_t1.3_p0.99_k128": (1.3, 0.99, 128),    # the policy-step parameters
    "top_k_only_t1.0_k50": (1.0, 1.0, 50),
    "wide_top_p_t1.3_p0.99": (1.3, 0.99, -1),           # tens of thousands of candidates
    "wide_top_k_k5000_p0.9": (1.0, 0.9, 5000),          # k beyond the tile-maximum bound
}


@pytest.mark.parametrize("name", list(CONFIGS))
def test_linear_pair_matches_oracle(name):
    tau, p, k = CONFIGS[name]
    T, H = 130, 256                                    # a ragged last row tile
    h, w, hb, wb, x, S, tg, full, restr, sup = _run(T, H, 100 + len(name), tau, p, k)
    check_pair("linear_pair_" + name, hb, wb, x, S, H, tau, p, k, tg, full, restr, sup)


def test_linear_pair_mixed_per_row_parameters():
    """Per-row tau, top-p and top-k from the rollout mix (tau > 0: no greedy rows here)."""
    T, H = 260, 256
    rng = np.random.default_rng(5)
    taus = rng.choice([0.7, 1.0, 1.3], T).astype(np.float32)
    ps = rng.choice([0.9, 0.95, 1.0], T).astype(np.float32)
    ks = rng.choice([-1, 50, 128], T).astype(np.int32)
    h, w, hb, wb, x, S, tg, full, restr, sup = _run(T, H, 6, taus, ps, ks)
    check_pair("linear_pair_mixed", hb, wb, x, S, H, taus, ps, ks, tg, full, restr, sup)


def test_linear_pair_full_equals_linear_logp_and_filters_off():
    """out_full is rlk_linear_logp's bit for bit; p = 1, k = -1 gives restr == full, support V."""
    h, w = _case(200, 512, 8)
    tg = torch.randint(0, VR, (200,), device=DEV, dtype=torch.int32)
    ref = pkg.linear_logp(h, w, tg, 1.1)
    full, restr, sup = pkg.linear_logp_pair(h, w, tg, 1.1, 1.0, -1)
    full2, _, _ = pkg.linear_logp_pair(h, w, tg, 1.1, 0.9, 64)
    torch.cuda.synchronize()
    assert torch.equal(full.view(torch.int32), ref.view(torch.int32))
    assert torch.equal(full2.view(torch.int32), ref.view(torch.int32))
    assert torch.equal(restr.view(torch.int32), full.view(torch.int32))
    assert (sup == VR).all()


def test_linear_pair_is_batch_invariant():
    """A row's bits do not depend on the batch: its row tile, the rows around
    it, or the other rows' parameters (which change how many rounds run)."""
    T, H = 300, 256
    h, w = _case(T, H, 9)
    g = torch.Generator(device=DEV).manual_seed(3)
    tg = torch.randint(0, VR, (T,), generator=g, device=DEV, dtype=torch.int32)
    taus = torch.full((T,), 1.3, device=DEV)
    ps = torch.full((T,), 0.95, device=DEV)
    ks = torch.full((T,), 128, dtype=torch.int32, device=DEV)
    a = pkg.linear_logp_pair(h, w, tg, taus, ps, ks)
    sub = torch.as_tensor([299, 5, 128, 127, 200, 0], device=DEV)
    big = torch.full((10, H + 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    big[4:, :H] = h[sub]
    b = pkg.linear_logp_pair(big[4:, :H], w, tg[sub].contiguous(), taus[sub].contiguous(),
                             ps[sub].contiguous(), ks[sub].contiguous())
    # the same rows among wide top-p rows (more rounds for the others)
    ps2 = torch.full((T,), 0.999, device=DEV)
    ks2 = torch.full((T,), -1, dtype=torch.int32, device=DEV)
    ps2[sub], ks2[sub] = 0.95, 128
    c = pkg.linear_logp_pair(h, w, tg, taus, ps2, ks2)
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(a[i][sub].view(torch.int32), b[i].view(torch.int32))
        assert torch.equal(a[i][sub].view(torch.int32), c[i][sub].view(torch.int32))


def test_linear_pair_edge_cases():
    """Uniform rows keep every tie; k = 1 keeps the maximum (restr 0 at the
    argmax); p below the top token's mass keeps one token; k = V is off."""
    H = 256
    h, w = _case(8, H, 10, hot=False)
    w[:, :] = 0.0                                      # every logit 0: all tied
    tg = torch.arange(8, device=DEV, dtype=torch.int32) * 1000
    full, restr, sup = pkg.linear_logp_pair(h, w, tg, 0.8, 0.3, 7)
    torch.cuda.synchronize()
    assert (sup == VR).all()
    assert torch.allclose(restr, torch.full_like(restr, -math.log(VR)), atol=2e-5)

    h, w = _case(64, H, 11)
    hb, wb = _bits(h), _bits(w)
    x, S = _exact_logits(hb, wb)
    am = torch.as_tensor(np.argmax(x, axis=1).astype(np.int32), device=DEV)
    f1, r1, s1 = pkg.linear_logp_pair(h, w, am, 1.0, 1.0, 1)
    f2, r2, s2 = pkg.linear_logp_pair(h, w, am, 1.0, 1e-3, -1)
    f3, r3, s3 = pkg.linear_logp_pair(h, w, am, 1.0, 1.0, VR)
    torch.cuda.synchronize()
    top2 = np.sort(x, axis=1)[:, -2:]
    clear = torch.as_tensor(top2[:, 1] - top2[:, 0] > 1e-3, device=DEV)   # no near-tie at the top
    assert clear.sum() > 32
    for s_, r_ in ((s1, r1), (s2, r2)):
        assert (s_[clear] == 1).all() and (r_[clear] == 0).all()
    assert (s3 == VR).all() and torch.equal(r3.view(torch.int32), f3.view(torch.int32))


def test_linear_pair_near_one_top_p_searches_every_key():
    """p within 1e-4 of 1: no a-priori window, the search starts over every key."""
    T, H = 40, 256
    h, w, hb, wb, x, S, tg, full, restr, sup = _run(T, H, 12, 1.3, 0.99995, -1, hot=False)
    check_pair("linear_pair_p0.99995", hb, wb, x, S, H, 1.3, 0.99995, -1, tg, full, restr, sup)


def test_linear_pair_rejected_and_nonfinite_rows():
    H = 256
    h, w = _case(8, H, 13)
    tg = torch.randint(0, VR, (8,), device=DEV, dtype=torch.int32)
    taus = torch.tensor([1.0, 0.0, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0], device=DEV)
    ps = torch.tensor([0.9, 0.9, 0.0, 1.5, 0.9, 0.9, 0.9, 0.9], device=DEV)
    ks = torch.tensor([50, 50, 50, 50, 0, -3, 50, 50], dtype=torch.int32, device=DEV)
    tg[6] = VR
    h[7, 3] = float("nan")
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    full, restr, sup = pkg.linear_logp_pair(h, w, tg, taus, ps, ks, err_count=err)
    torch.cuda.synchronize()
    f, r, s = full.cpu().numpy(), restr.cpu().numpy(), sup.cpu().numpy()
    assert err.item() == 6
    for i in range(1, 8):
        assert math.isnan(r[i]) and s[i] == -1, i
    assert all(math.isnan(f[i]) for i in range(1, 8))
    assert math.isfinite(f[0]) and math.isfinite(r[0]) or r[0] == -math.inf
    assert 1 <= s[0] <= VR


def test_linear_pair_full_size_sampled_rows():
    """T = 8192, H = 4096 (the bench's case): the policy-step parameters (tau
    1.3, top-p 0.99, top-k 128; rows listed from the kept logits) and top-p
    alone at tau 1.0, p 0.95 (GEMM window rounds); every output finite, sampled
    rows against the oracle."""
    T, H = 8192, 4096
    h, w = _case(T, H, 14)
    g = torch.Generator(device=DEV).manual_seed(15)
    tg = torch.randint(0, VR, (T,), generator=g, device=DEV, dtype=torch.int32)
    rows = np.array([0, 1, 127, 128, 4095, 4096, 8190, 8191])
    ri = torch.as_tensor(rows, device=DEV)
    hb, wb = _bits(h[ri]), _bits(w)
    x, S = _exact_logits(hb, wb)
    for name, (tau, p, k) in (("policy_step", (1.3, 0.99, 128)), ("top_p_only", (1.0, 0.95, -1))):
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        full, restr, sup = pkg.linear_logp_pair(h, w, tg, tau, p, k, err_count=err)
        torch.cuda.synchronize()
        assert err.item() == 0 and torch.isfinite(full).all() and (sup >= 1).all(), name
        check_pair("linear_pair_full_size_" + name, hb, wb, x, S, H, tau, p, k, tg.cpu().numpy()[rows],
                   full.cpu().numpy()[rows], restr.cpu().numpy()[rows], sup.cpu().numpy()[rows])
    del h, w
    torch.cuda.empty_cache()
