"""GPU parity: the CUDA path against the CPU oracle, element by element.

Tolerance: |delta logprob| <= 2e-5 absolute on both outputs; supports equal,
except at tie classes whose renormalised mass above them lies within 1e-6
(relative) of p, which are counted and then scored on the support the GPU
chose.  All calls go through the C ABI (the ctypes binding).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import rollout_consistent_vocab_gb300 as pkg
from rollout_consistent_vocab_gb300 import workloads as W

from _support import (TOL, Stats, bits_of, check_row, check_rows, check_rows_parallel,
                      oracle_targets, oracle_targets_parallel, record)

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


def run_pair(x, t, tau, p, k):
    full, restr, sup = pkg.logp_pair(x, t, tau, p, k)
    torch.cuda.synchronize()
    return full.cpu().numpy(), restr.cpu().numpy(), sup.cpu().numpy()


def rows_from_bits(rows_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(rows_bits.view(np.int16).copy()).to(DEV).view(torch.bfloat16)


# ------------------------------------------------------------------ golden

def test_golden_tiny16():
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny16.json")
    data = json.load(open(path))
    dec = lambda v: -math.inf if v == "-inf" else float(v)
    for case in data["cases"]:
        row = np.full(VP, 0xFF80, dtype=np.uint16)
        vals = np.asarray(case["values"], dtype=np.float32)
        row[case["cols"]] = (vals.view(np.uint32) >> 16).astype(np.uint16)
        targets = [pt[0] for pt in case["per_target"]]
        x = rows_from_bits(np.stack([row] * len(targets)))
        f, r, s = run_pair(x, _t(targets, torch.int32), case["tau"], case["top_p"], case["top_k"])
        for i, (t, full, restr, sup) in enumerate(case["per_target"]):
            assert f[i] == dec(full) or abs(f[i] - dec(full)) <= TOL, (case["tau"], t)
            assert r[i] == dec(restr) or abs(r[i] - dec(restr)) <= TOL, (case, t)
            assert s[i] == sup


# ------------------------------------------------------------------ pins on the GPU

def _row(fill, values=None, pad="neginf"):
    import test_oracle_pins as P
    return P.make_row(fill, values, pad)


def test_pins_uniform_dominant_two_valued():
    rows = [_row(1.5), _row(-64.0, {77: 64.0}),
            _row(0.0, {j: 12.0 for j in range(1000, 1000 + 32 * 97, 97)})]
    x = rows_from_bits(np.stack(rows))
    t = _t([5, 77, 1000 + 3 * 97], torch.int32)
    f, r, s = run_pair(x, t, _t([0.7, 1.0, 0.7], torch.float32), _t([0.95, 0.95, 0.95], torch.float32),
                       _t([-1, -1, -1], torch.int32))
    assert abs(f[0] - (-math.log(VR))) <= TOL and abs(r[0] - (-math.log(VR))) <= TOL and s[0] == VR
    assert abs(f[1]) <= TOL and r[1] == 0.0 and s[1] == 1
    hs = float(np.float32(12.0) / np.float32(0.7))
    assert abs(f[2] - (-math.log(32 + (VR - 32) * math.exp(-hs)))) <= TOL
    assert abs(r[2] - (-math.log(32))) <= TOL and s[2] == 32
    # top-k 50 on the uniform row keeps every tied token
    f, r, s = run_pair(x[:1], t[:1], 1.3, 0.99, 50)
    assert s[0] == VR and abs(r[0] + math.log(VR)) <= TOL


def test_pins_staircase_and_order():
    row = _row(-128.0, {j: -float(j) for j in range(64)})
    x = rows_from_bits(np.stack([row] * 4))
    t = _t([0, 2, 0, 1], torch.int32)
    f, r, s = run_pair(x, t, 1.0, _t([0.95, 0.95, 0.7, 0.75], torch.float32),
                       _t([-1, -1, 2, 2], torch.int32))
    assert s[0] == 3 and abs(r[0] - (-0.4076059644443804)) <= TOL
    assert abs(f[0] - (-0.45867514538708193)) <= TOL
    assert abs(r[1] - (-2 - math.log(1 + math.exp(-1) + math.exp(-2)))) <= TOL
    assert s[2] == 1 and r[2] == 0.0
    assert s[3] == 2 and abs(r[3] - (-1 - math.log(1 + math.exp(-1)))) <= TOL


def test_pins_topk1_ties_greedy():
    rng = np.random.default_rng(11)
    cols = rng.choice(VR, 50, replace=False)
    vals = {int(j): float(v) for j, v in zip(cols, np.arange(1, 51, dtype=np.float32))}
    amax = max(vals, key=vals.get)
    rows = [_row(0.0, vals), _row(0.0, vals),
            _row(-20.0, {10: 3.0, 11: 2.0, 12: 1.0, 13: 1.0, 14: 1.0, 15: 1.0, 16: 1.0}),
            _row(0.0, {500: 7.0, 90000: 7.0, 3: 6.0}), _row(0.0, {500: 7.0, 90000: 7.0, 3: 6.0}),
            _row(0.0, {150000: 9.0, 151935: 9.0})]
    x = rows_from_bits(np.stack(rows))
    t = _t([amax, (amax + 1) % VR, 16, 500, 90000, 150000], torch.int32)
    f, r, s = run_pair(x, t, _t([0.9, 0.9, 1.0, 0.0, 0.0, 0.0], torch.float32),
                       _t([0.5, 1.0, 1.0, 0.9, 0.9, 1.0], torch.float32),
                       _t([1, 1, 3, 50, 50, -1], torch.int32))
    assert r[0] == 0.0 and s[0] == 1 and r[1] == -math.inf
    assert s[2] == 7 and abs(r[2] - (1 - math.log(math.exp(3) + math.exp(2) + 5 * math.exp(1)))) <= TOL
    assert f[3] == 0.0 and r[3] == 0.0 and f[4] == -math.inf and r[4] == -math.inf
    assert f[5] == 0.0 and s[5] == 1


def test_padding_is_ignored_and_nonfinite_rows():
    base = {j: float(j % 13) for j in range(0, VR, 1237)}
    rows = [_row(-3.0, base, "neginf"), _row(-3.0, base, "garbage")]
    nan_row = _row(-3.0, base)
    nan_row[777] = 0x7FC0
    inf_row = _row(-3.0, base)
    inf_row[151935] = 0x7F80
    allneg = _row(float("-inf"))
    two = _row(float("-inf"), {7: 0.0, 8: 0.0})
    nan_chunk = _row(-3.0, base)
    nan_chunk[800:808] = 0x7FC1          # a whole 16-byte chunk of NaN
    x = rows_from_bits(np.stack(rows + [nan_row, inf_row, allneg, two, two, nan_chunk]))
    t = _t([1237, 1237, 1237, 1237, 0, 7, 9, 1237], torch.int32)
    f, r, s = run_pair(x, t, 0.9, 0.9, 64)
    assert f[0] == f[1] and r[0] == r[1] and s[0] == s[1]
    for i in (2, 3, 4, 7):
        assert math.isnan(f[i]) and math.isnan(r[i]) and s[i] == -1, i
    assert abs(f[5] + math.log(2)) <= TOL and f[6] == -math.inf
    # full-only and greedy on NaN rows are NaN too
    f1 = pkg.logp_full(x, t, 0.9)
    torch.cuda.synchronize()
    assert all(math.isnan(f1[i].item()) for i in (2, 3, 4, 7))
    sel = [2, 3, 4, 7]
    f, r, s = run_pair(x[sel], t[sel], 0.0, 1.0, -1)
    assert all(math.isnan(v) for v in f) and all(v == -1 for v in s)


def test_invalid_per_row_parameters_are_counted():
    x, hot, n = W.hot_logits(8, 4, 8, seed=5, device=DEV)
    t = W.structural_targets(8, hot, n, seed=5, device=DEV)
    t[7] = VR        # out of range target
    tau = _t([0.7, -1.0, float("nan"), 0.7, 0.7, 0.7, 0.7, 0.7], torch.float32)
    p = _t([0.9, 0.9, 0.9, 0.0, 1.5, 0.9, 0.9, 0.9], torch.float32)
    k = _t([-1, -1, -1, -1, -1, 0, VR + 1, -1], torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    f, r, s = pkg.logp_pair(x, t, tau, p, k, err_count=err)
    torch.cuda.synchronize()
    assert err.item() == 7
    assert not math.isnan(f[0].item()) and s[0].item() > 0
    assert torch.isnan(f[1:]).all() and torch.isnan(r[1:]).all() and (s[1:] == -1).all()


# ------------------------------------------------------------------ the workloads

def test_c0_spread_all_rows():
    """64 rows of N(0,3^2), tau 0.7, p 0.95; oracle targets, 4 rows forced outside."""
    wl = W.workload_c0(device=DEV)
    bits = bits_of(wl.logits)
    rng = np.random.default_rng(0)
    forced = set(rng.choice(wl.T, 4, replace=False).tolist())
    ones = np.ones(wl.T)
    targets = oracle_targets(bits, 0.7 * ones, 0.95 * ones, -ones.astype(int), rng, forced)
    f, r, s = run_pair(wl.logits, _t(targets, torch.int32), 0.7, 0.95, -1)
    st = Stats()
    check_rows(st, bits, 0.7 * ones, 0.95 * ones, -ones, targets, f, r, s)
    assert sum(r[i] == -math.inf for i in forced) == 4
    record("c0 T=64 N(0,9) tau0.7 p0.95", st)


def test_c1_microbatch_all_rows():
    """T = 1024 rows, every row checked: targets drawn from each row's restricted
    distribution by the oracle, 5% of the rows forced outside the support."""
    wl = W.workload_c1(device=DEV)
    T = wl.T
    bits = bits_of(wl.logits)
    rng = np.random.default_rng(1)
    forced = np.zeros(T, bool)
    forced[rng.choice(T, T // 20, replace=False)] = True
    tg = oracle_targets_parallel(bits, 0.7, 0.95, -1, forced, seed=1)
    f, r, s = run_pair(wl.logits, _t(tg, torch.int32), 0.7, 0.95, -1)
    st = Stats()
    check_rows_parallel(st, bits, 0.7, 0.95, -1, tg, f, r, s)
    assert st.rows == T
    assert np.all(r[forced] == -np.inf)
    record("c1 T=1024 hot32 tau0.7 p0.95", st, forced_out=int(forced.sum()))


def test_c2_pair_and_kl_all_rows():
    """T = 8192, tau 1.3, p 0.99, k 128, plus the KL term against perturbed
    reference logits; every row's pair, reference full logprob and KL term
    checked (targets from the oracle's restricted distribution, 5% forced out)."""
    wl = W.workload_c2(device=DEV)
    T = wl.T
    bits = bits_of(wl.logits)
    rbits = bits_of(wl.ref_logits)
    rng = np.random.default_rng(2)
    forced = np.zeros(T, bool)
    forced[rng.choice(T, T // 20, replace=False)] = True
    tg_np = oracle_targets_parallel(bits, 1.3, 0.99, 128, forced, seed=2)
    targets = _t(tg_np, torch.int32)
    full, restr, sup, full_ref, kl = pkg.logp_kl(wl.logits, wl.ref_logits, targets, 1.3, 0.99, 128)
    f2, r2, s2 = pkg.logp_pair(wl.logits, targets, 1.3, 0.99, 128)
    torch.cuda.synchronize()
    assert torch.equal(full, f2) and torch.equal(restr.nan_to_num(), r2.nan_to_num()) and torch.equal(sup, s2)
    assert torch.equal(kl, full - full_ref)
    f, r, s = full.cpu().numpy(), restr.cpu().numpy(), sup.cpu().numpy()
    st = Stats()
    check_rows_parallel(st, bits, 1.3, 0.99, 128, tg_np, f, r, s, ref_bits=rbits,
                        full_ref=full_ref.cpu().numpy(), kl=kl.cpu().numpy())
    assert st.rows == T
    assert (s >= 1).all() and (s <= 128 + 64).all()
    assert np.all(r[forced] == -np.inf)
    record("c2 T=8192 hot1-256 tau1.3 p0.99 k128 (+ref, kl)", st, forced_out=int(forced.sum()))


def test_c4_mixed_parameters_all_rows():
    """T = 55296 (16.9 GB of logits) with per-row tau/p/k: every row checked,
    in blocks of 4096 rows copied to the host."""
    wl = W.workload_c4(device=DEV)
    T = wl.T
    targets = W.structural_targets(T, wl.hot, wl.hot_n, seed=4, device=DEV)
    full, restr, sup = pkg.logp_pair(wl.logits, targets, wl.temperature, wl.top_p, wl.top_k)
    torch.cuda.synchronize()
    tau, p, k = wl.temperature.cpu().numpy(), wl.top_p.cpu().numpy(), wl.top_k.cpu().numpy()
    f, r, s, tg = full.cpu().numpy(), restr.cpu().numpy(), sup.cpu().numpy(), targets.cpu().numpy()
    st = Stats()
    for a in range(0, T, 4096):
        b = min(T, a + 4096)
        bits = bits_of(wl.logits[a:b])
        check_rows_parallel(st, bits, tau[a:b], p[a:b], k[a:b], tg[a:b], f[a:b], r[a:b], s[a:b],
                            rows=np.arange(a, b))
    assert st.rows == T
    kinds = {}
    for tv in np.unique(tau):
        for pv in np.unique(p):
            for kv in np.unique(k):
                kinds[f"{tv:g}/{pv:g}/{kv}"] = int(np.sum((tau == tv) & (p == pv) & (k == kv)))
    record("c4 T=55296 mixed tau/p/k", st, rows_per_kind=kinds)
    del wl, full, restr, sup
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [1, 7, 300])
def test_ragged_batches_random_parameters(T):
    rng = np.random.default_rng(T)
    x, hot, n = W.hot_logits(T, 1, 300, seed=100 + T, device=DEV)
    tau = rng.choice([0.0, 0.5, 0.7, 1.0, 1.3, 2.0], T).astype(np.float32)
    p = rng.choice([0.3, 0.8, 0.9, 0.95, 0.99, 0.9999, 1.0], T).astype(np.float32)
    k = rng.choice([-1, 1, 5, 50, 128, 256, 257, 1000], T).astype(np.int32)
    bits = bits_of(x)
    forced = set(rng.choice(T, max(1, T // 10), replace=False).tolist())
    tg = oracle_targets(bits, tau, p, k, rng, forced)
    f, r, s = run_pair(x, _t(tg, torch.int32), _t(tau, torch.float32), _t(p, torch.float32),
                       _t(k, torch.int32))
    st = Stats()
    check_rows(st, bits, tau, p, k, tg, f, r, s)
    record(f"ragged T={T} random tau/p/k", st)


def test_entry_points_agree_bitwise():
    x, hot, n = W.hot_logits(64, 1, 256, seed=9, device=DEV)
    t = W.structural_targets(64, hot, n, seed=9, device=DEV)
    f, r, s = pkg.logp_pair(x, t, 1.3, 0.99, 128)
    f1 = pkg.logp_full(x, t, 1.3)
    r1, s1 = pkg.logp_restricted(x, t, 1.3, 0.99, 128)
    torch.cuda.synchronize()
    assert torch.equal(f, f1) and torch.equal(r, r1) and torch.equal(s, s1)


def test_row_stride_and_buffer_offset():
    """Rows inside a wider buffer (row stride 152576 + 8j) give the same bits."""
    x, hot, n = W.hot_logits(33, 1, 64, seed=13, device=DEV)
    t = W.structural_targets(33, hot, n, seed=13, device=DEV)
    f0, r0, s0 = pkg.logp_pair(x, t, 0.7, 0.95, -1)
    for extra in (8, 64, 4096):
        big = torch.full((33 + 3, VP + extra), float("nan"), dtype=torch.bfloat16, device=DEV)
        big[3:, :VP] = x
        f1, r1, s1 = pkg.logp_pair(big[3:], t, 0.7, 0.95, -1)
        torch.cuda.synchronize()
        assert torch.equal(f0, f1) and torch.equal(r0, r1) and torch.equal(s0, s1)


def test_top_p_only_deep_nucleus():
    """Top-p without top-k, p close to 1, on spread and on hot rows: the candidate
    window derived from the total mass must still hold the whole nucleus."""
    rng = np.random.default_rng(55)
    xs = W.spread_logits(6, 2.0, seed=55, device=DEV)
    xh, hot, n = W.hot_logits(6, 1, 64, seed=56, device=DEV)
    x = torch.cat([xs, xh])
    T = x.shape[0]
    tau = rng.choice([0.7, 1.0, 1.3], T).astype(np.float32)
    p = rng.choice([0.99, 0.999, 0.9999, 0.99999], T).astype(np.float32)
    k = np.full(T, -1, np.int32)
    bits = bits_of(x)
    tg = oracle_targets(bits, tau, p, k, rng, {0, 7})
    f, r, s = run_pair(x, _t(tg, torch.int32), _t(tau, torch.float32), _t(p, torch.float32),
                       _t(k, torch.int32))
    st = Stats()
    check_rows(st, bits, tau, p, k, tg, f, r, s)
    record("deep nucleus top-p only", st)


def test_wide_support_fallback_path():
    """Supports reaching more than 1024 order keys below the maximum take the
    global-memory window path; still exact against the oracle."""
    rng = np.random.default_rng(77)
    T = 6
    # logits centred on 0 with small spread: the nucleus crosses zero
    x = (0.02 * rng.standard_normal((T, VP))).astype(np.float32)
    x[:, 5] = 3.0
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    bits[:, VR:] = 0xFF80
    tau = np.array([1.0, 1.0, 0.5, 1.0, 2.0, 1.0], np.float32)
    p = np.array([0.9, 0.5, 0.99, 1.0, 0.7, 0.99], np.float32)
    k = np.array([-1, -1, -1, 100000, 70000, 3000], np.int32)
    forced = {1}
    tg = oracle_targets(bits, tau, p, k, rng, forced)
    f, r, s = run_pair(rows_from_bits(bits), _t(tg, torch.int32), _t(tau, torch.float32),
                       _t(p, torch.float32), _t(k, torch.int32))
    st = Stats()
    check_rows(st, bits, tau, p, k, tg, f, r, s)
    record("wide support (global-memory windows)", st)


def test_window_reaching_minus_infinity():
    """Rows whose maximum lies within a few order keys of -inf and whose top-k
    witness is -inf: the candidate window then reaches -inf itself, and only
    the shard's real chunks may be counted (the support includes the -inf
    tokens, at zero mass).  Also drawn, through both sampler paths."""
    rng = np.random.default_rng(91)
    rows, first = [], []
    for n_fin in (100, 3, 5000):
        cols = rng.choice(VR, n_fin, replace=False)
        vals = rng.choice([-1.75 * 2.0 ** 127, -1.5 * 2.0 ** 127, -1.25 * 2.0 ** 127], n_fin)
        rows.append(_row(float("-inf"), {int(c): float(v) for c, v in zip(cols, vals)}, "garbage"))
        first.append(int(cols[np.argmax(vals)]))
    bits = np.stack(rows * 3)
    x = rows_from_bits(bits)
    T = bits.shape[0]
    taus = np.array([1.0] * T, np.float32)
    ps = np.array([1.0, 1.0, 1.0, 0.9, 0.9, 0.9, 0.9, 0.9, 0.9], np.float32)
    ks = np.array([1000, 1000, 1000, 1000, 1000, 1000, -1, -1, -1], np.int32)
    ts = np.array(first * 3, np.int32)
    ts[1] = 5                                   # a -inf column
    f, r, s = run_pair(x, _t(ts, torch.int32), _t(taus, torch.float32), _t(ps, torch.float32),
                       _t(ks, torch.int32))
    st = Stats()
    check_rows(st, bits, taus, ps, ks, ts, f, r, s)
    u = torch.as_tensor(rng.integers(0, 2 ** 32, T, dtype=np.uint64).astype(np.uint32).view(np.int32),
                        device=DEV)
    tok, rs, fs, ss = pkg.sample(x, _t(taus, torch.float32), _t(ps, torch.float32), _t(ks, torch.int32),
                                 uniform=u)
    torch.cuda.synchronize()
    for i in range(T):
        o = oracle.logp_row(bits[i], float(taus[i]), float(ps[i]), int(ks[i]), int(tok[i]))
        assert math.isfinite(o.restr) and int(ss[i]) == o.support, i


def test_top_p_only_high_temperature_rows_all_checked():
    """Top-p-only rows at temperatures 1.0 and 1.3 (p 0.9 .. 0.99, k off) on
    hot-set logits: the rows with the widest candidate windows (tens of
    thousands of candidates each).  Every row against the oracle (targets from the oracle's
    restricted distribution, a tenth forced outside the support)."""
    T = 384
    rng = np.random.default_rng(21)
    x, hot, n = W.hot_logits(T, 1, 512, seed=21, device=DEV)
    tau = rng.choice([1.0, 1.3], T).astype(np.float32)
    p = rng.choice([0.9, 0.95, 0.97, 0.99], T).astype(np.float32)
    k = np.full(T, -1, np.int32)
    bits = bits_of(x)
    forced = np.zeros(T, bool)
    forced[rng.choice(T, T // 10, replace=False)] = True
    tg = oracle_targets_parallel(bits, tau, p, k, forced, seed=21)
    f, r, s = run_pair(x, _t(tg, torch.int32), _t(tau, torch.float32), _t(p, torch.float32),
                       _t(k, torch.int32))
    st = Stats()
    check_rows_parallel(st, bits, tau, p, k, tg, f, r, s)
    assert st.rows == T
    record("top-p only tau1.0/1.3 p0.9-0.99 hot1-512", st)


def test_negative_logit_rows_dense_windows():
    """Hot-set logits shifted by -40, so every logit of a row is negative (the
    row maximum about -16): at temperature 1.3 and top-p 0.99 the candidate
    window holds tens of thousands of negative values and is counted by the
    dense form's general branch (order keys of negative values), at p 0.9 and
    with top-k 128 by the sparser paths.  Every row against the oracle."""
    T = 256
    rng = np.random.default_rng(23)
    x, hot, n = W.hot_logits(T, 1, 512, seed=23, device=DEV)
    x = (x.float() - 40.0).to(torch.bfloat16)
    tau = rng.choice([1.0, 1.3], T).astype(np.float32)
    p = rng.choice([0.9, 0.99], T).astype(np.float32)
    k = rng.choice([-1, -1, 128], T).astype(np.int32)
    bits = bits_of(x)
    assert ((bits[:, :VR] & 0x8000) != 0).all()      # every real logit negative
    forced = np.zeros(T, bool)
    forced[rng.choice(T, T // 10, replace=False)] = True
    tg = oracle_targets_parallel(bits, tau, p, k, forced, seed=23)
    f, r, s = run_pair(x, _t(tg, torch.int32), _t(tau, torch.float32), _t(p, torch.float32),
                       _t(k, torch.int32))
    st = Stats()
    check_rows_parallel(st, bits, tau, p, k, tg, f, r, s)
    assert st.rows == T
    record("negative logits tau1.0/1.3 p0.9/0.99 k off/128", st)


def test_extreme_temperatures_all_rows():
    """Temperatures far from 1 (1e-3, 0.05, 5, 50) with top-p 0.5 .. 1 and
    top-k off, 1, 7, 1000: near-greedy rows whose masses underflow to the
    maximum's ties, and near-flat rows whose nucleus reaches below the first
    window (the global-memory windows).  Every row against the oracle; the
    tolerance adds 2.4e-7 max(|M|, |x_t|) / tau to 2e-5: at temperature 1e-3
    the scaled logits reach about 2.4e4, and float32 holds each to a relative
    2^-24 (the oracle rounds every x / tau, the kernel (x_t - M) / tau), four
    such roundings at most."""
    T = 128
    rng = np.random.default_rng(29)
    x, hot, n = W.hot_logits(T, 1, 64, seed=29, device=DEV)
    tau = rng.choice([1e-3, 0.05, 5.0, 50.0], T).astype(np.float32)
    p = rng.choice([0.5, 0.9, 0.999, 1.0], T).astype(np.float32)
    k = rng.choice([-1, 1, 7, 1000], T).astype(np.int32)
    bits = bits_of(x)
    forced = np.zeros(T, bool)
    forced[rng.choice(T, T // 10, replace=False)] = True
    tg = oracle_targets_parallel(bits, tau, p, k, forced, seed=29)
    f, r, s = run_pair(x, _t(tg, torch.int32), _t(tau, torch.float32), _t(p, torch.float32),
                       _t(k, torch.int32))
    st = Stats()
    check_rows_parallel(st, bits, tau, p, k, tg, f, r, s, scale_tol=2.4e-7)
    assert st.rows == T
    record("extreme temperatures 1e-3..50, p 0.5..1, k off/1/7/1000", st)


def test_coarse_ties_all_rows():
    """Logits quantised to 17 values (multiples of 0.5 in [-4, 4]): every
    threshold falls inside a tie class of thousands of tokens, so the
    top-k support (ties kept) is far larger than k and the nucleus takes or
    drops whole classes.  Every row against the oracle."""
    T = 96
    rng = np.random.default_rng(31)
    g = torch.Generator(device=DEV).manual_seed(31)
    x = torch.full((T, VP), float("-inf"), device=DEV)
    x[:, :VR] = torch.clamp(torch.round(2.0 * torch.randn((T, VR), generator=g, device=DEV)) / 2.0, -4.0, 4.0)
    x = x.to(torch.bfloat16)
    tau = rng.choice([0.7, 1.0, 1.3], T).astype(np.float32)
    p = rng.choice([0.5, 0.9, 0.99, 1.0], T).astype(np.float32)
    k = rng.choice([-1, 1, 10, 1000, 50000], T).astype(np.int32)
    bits = bits_of(x)
    forced = np.zeros(T, bool)
    forced[rng.choice(T, T // 10, replace=False)] = True
    tg = oracle_targets_parallel(bits, tau, p, k, forced, seed=31)
    f, r, s = run_pair(x, _t(tg, torch.int32), _t(tau, torch.float32), _t(p, torch.float32),
                       _t(k, torch.int32))
    st = Stats()
    check_rows_parallel(st, bits, tau, p, k, tg, f, r, s)
    assert st.rows == T
    record("coarse ties: 17 values, tau 0.7-1.3, p 0.5-1, k off/1/10/1000/50000", st)
