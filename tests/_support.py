"""Shared helpers of the GPU parity tests (these may call the oracle)."""

import math

import numpy as np
import torch

import oracle

TOL = 2e-5          # |delta logprob| bound against the oracle
MARGIN = 1e-6       # relative distance of a tie class to the nucleus threshold that may differ


def bits_of(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def param_at(v, i):
    if isinstance(v, torch.Tensor):
        return v[i].item()
    if isinstance(v, np.ndarray):
        return v[i].item()
    return v


def oracle_targets(bits_rows: np.ndarray, taus, ps, ks, rng: np.random.Generator,
                   forced_out: set) -> np.ndarray:
    """Targets drawn from each row's restricted distribution (oracle), or uniformly
    from the real tokens outside the support for rows in ``forced_out``."""
    out = np.empty(bits_rows.shape[0], dtype=np.int32)
    for n in range(bits_rows.shape[0]):
        tau, p, k = taus[n], ps[n], ks[n]
        if tau == 0.0:
            x = oracle.bf16_bits_to_f32(bits_rows[n][:oracle.VREAL])
            a = int(np.argmax(x))
            out[n] = a if n not in forced_out else (a + 1 + rng.integers(oracle.VREAL - 1)) % oracle.VREAL
            continue
        _, restr, S = oracle.row_logprobs_all(bits_rows[n], tau, p, k)
        if n in forced_out:
            outside = np.nonzero(~S)[0]
            out[n] = int(rng.choice(outside)) if len(outside) else int(rng.integers(oracle.VREAL))
        else:
            w = np.exp(restr[S] - restr[S].max())
            out[n] = int(rng.choice(np.nonzero(S)[0], p=w / w.sum()))
    return out


class Stats:
    def __init__(self):
        self.rows = 0
        self.near_threshold = 0
        self.max_full = 0.0
        self.max_restr = 0.0

    def __repr__(self):
        return (f"rows={self.rows} near_threshold={self.near_threshold} "
                f"max|dfull|={self.max_full:.3g} max|drestr|={self.max_restr:.3g}")


def _close(a: float, b: float, tol: float) -> bool:
    if math.isnan(b):
        return math.isnan(a)
    if math.isinf(b):
        return a == b
    return abs(a - b) <= tol


def check_row(stats: Stats, bits_row, tau, p, k, t, g_full, g_restr, g_sup, tol=TOL,
              check_full=True, check_restr=True):
    """Compare one row of GPU outputs with the oracle; returns the oracle result."""
    try:
        r = oracle.logp_row(bits_row, tau, p, k, t, want_margins=True)
    except oracle.InvalidArgument:
        assert math.isnan(g_full) or not check_full
        assert math.isnan(g_restr) or not check_restr
        return None
    stats.rows += 1
    ctx = f"tau={tau} p={p} k={k} t={t}"
    if check_full:
        assert _close(g_full, r.full, tol), f"full {g_full} vs {r.full} ({ctx})"
        if math.isfinite(r.full):
            stats.max_full = max(stats.max_full, abs(g_full - r.full))
    if not check_restr:
        return r
    want_restr = r.restr
    if g_sup != r.support:
        # allowed only at tie classes within MARGIN of the nucleus threshold
        assert r.g_desc is not None, f"support {g_sup} vs {r.support} with top-p off ({ctx})"
        cum = np.cumsum(r.counts_desc)
        assert g_sup in cum, f"support {g_sup} is not a tie-class boundary ({ctx})"
        j_g = int(np.nonzero(cum == g_sup)[0][0])
        j_o = int(np.nonzero(cum == r.support)[0][0])
        lo_j, hi_j = min(j_g, j_o) + 1, max(j_g, j_o)
        for j in range(lo_j, hi_j + 1):
            rel = abs(r.g_desc[j] - p) / p
            assert rel <= MARGIN, f"class {j} margin {rel:.3g} > {MARGIN} ({ctx})"
        stats.near_threshold += 1
        want_restr = oracle.restr_for_support_size(bits_row, tau, t, int(g_sup))
    assert _close(g_restr, want_restr, tol), f"restr {g_restr} vs {want_restr} ({ctx})"
    if math.isfinite(want_restr):
        stats.max_restr = max(stats.max_restr, abs(g_restr - want_restr))
    return r


def check_rows(stats, x_rows_bits, taus, ps, ks, ts, full, restr, sup, **kw):
    for n in range(x_rows_bits.shape[0]):
        check_row(stats, x_rows_bits[n], float(taus[n]), float(ps[n]), int(ks[n]), int(ts[n]),
                  float(full[n]), float(restr[n]), int(sup[n]), **kw)
