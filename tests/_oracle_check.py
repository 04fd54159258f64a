"""Row-by-row comparison of GPU outputs with the CPU oracle (test infrastructure).

This module imports numpy and the oracle only (no torch), so that it can run
in worker processes: ``check_rows_parallel`` and ``oracle_targets_parallel``
fan the oracle out over one spawned process per host core, which lets the
parity tests compare every row of the full-size workloads.

Tolerance: |delta logprob| <= 2e-5 absolute on both outputs.  Supports must
be equal, except at a tie class whose renormalised mass strictly above it
lies within 1e-6 (relative) of p: there both choices are correct to the
precision of the arithmetic, so such rows are counted, and scored on the
support the GPU chose.  Every row whose nucleus has a class that close to
the threshold is counted too (``near_rows``, and its tokens in
``near_tokens``), whether or not the GPU's support differs.
"""

from __future__ import annotations

import math
import multiprocessing as mp
import os

import numpy as np

import oracle

TOL = 2e-5          # |delta logprob| bound against the oracle
MARGIN = 1e-6       # relative distance of a tie class to the nucleus threshold that may differ
CHUNK = 16          # rows per worker task

# name -> summary dict of every comparison run in this process (printed at
# the end of the test session)
REPORT: dict = {}


class Stats:
    """Per-workload tally of a comparison."""

    FIELDS = ("rows", "near_rows", "near_tokens", "support_differs", "max_full", "max_restr",
              "max_kl")

    def __init__(self):
        self.rows = 0
        self.near_rows = 0          # rows with a tie class within MARGIN of the nucleus threshold
        self.near_tokens = 0        # tokens in those classes
        self.support_differs = 0    # rows where the GPU's support differs (all near the threshold)
        self.max_full = 0.0
        self.max_restr = 0.0
        self.max_kl = 0.0

    @property
    def near_threshold(self):
        return self.support_differs

    def merge(self, other: "Stats") -> "Stats":
        self.rows += other.rows
        self.near_rows += other.near_rows
        self.near_tokens += other.near_tokens
        self.support_differs += other.support_differs
        self.max_full = max(self.max_full, other.max_full)
        self.max_restr = max(self.max_restr, other.max_restr)
        self.max_kl = max(self.max_kl, other.max_kl)
        return self

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f in self.FIELDS}

    def __repr__(self):
        return (f"rows={self.rows} near_rows={self.near_rows} near_tokens={self.near_tokens} "
                f"support_differs={self.support_differs} max|dfull|={self.max_full:.3g} "
                f"max|drestr|={self.max_restr:.3g} max|dkl|={self.max_kl:.3g}")


def record(name: str, stats: Stats, **extra) -> None:
    """Keep a workload's tally for the end-of-session parity summary."""
    d = stats.as_dict() if isinstance(stats, Stats) else dict(stats)
    d.update(extra)
    REPORT[name] = d


def _close(a: float, b: float, tol: float) -> bool:
    if math.isnan(b):
        return math.isnan(a)
    if math.isinf(b):
        return a == b
    return abs(a - b) <= tol


def scaled_magnitude(bits_row, tau: float, t: int) -> float:
    """max(|M|, |x_t|) / tau over the real columns: the size of the scaled
    logits whose float32 rounding the logprobs inherit (0 for greedy rows)."""
    if not tau > 0.0:
        return 0.0
    x = oracle.bf16_bits_to_f32(np.asarray(bits_row)[:oracle.VREAL]).astype(np.float64)
    fin = x[np.isfinite(x)]
    m = float(np.max(np.abs(fin))) if fin.size else 0.0
    xt = float(x[t]) if math.isfinite(float(x[t])) else 0.0
    return max(m, abs(xt)) / float(np.float32(tau))


def check_row(stats: Stats, bits_row, tau, p, k, t, g_full, g_restr, g_sup, tol=TOL,
              check_full=True, check_restr=True, scale_tol=0.0):
    """Compare one row of GPU outputs with the oracle; returns the oracle result.
    ``scale_tol`` adds scale_tol * max(|M|, |x_t|) / tau to the tolerance: at
    temperatures far below 1 the scaled logits reach 1e4 and both sides
    round them (the oracle each s_j to float32, the kernel (x_t - M) / tau)."""
    if scale_tol > 0.0:
        tol = tol + scale_tol * scaled_magnitude(bits_row, tau, t)
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
    if r.g_desc is not None:
        rel = np.abs(r.g_desc - p) / p
        near = rel <= MARGIN
        if near.any():
            stats.near_rows += 1
            stats.near_tokens += int(np.sum(r.counts_desc[near]))
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
        stats.support_differs += 1
        want_restr = oracle.restr_for_support_size(bits_row, tau, t, int(g_sup))
    assert _close(g_restr, want_restr, tol), f"restr {g_restr} vs {want_restr} ({ctx})"
    if math.isfinite(want_restr):
        stats.max_restr = max(stats.max_restr, abs(g_restr - want_restr))
    return r


def check_rows(stats, x_rows_bits, taus, ps, ks, ts, full, restr, sup, **kw):
    for n in range(x_rows_bits.shape[0]):
        check_row(stats, x_rows_bits[n], float(taus[n]), float(ps[n]), int(ks[n]), int(ts[n]),
                  float(full[n]), float(restr[n]), int(sup[n]), **kw)


def target_row(bits_row, tau, p, k, forced_out: bool, seed) -> int:
    """A target drawn from the row's restricted distribution (oracle), or
    uniformly from the real tokens outside the support when ``forced_out``;
    greedy rows take the argmax (or, forced out, any other column)."""
    rng = np.random.default_rng(seed)
    if tau == 0.0:
        x = oracle.bf16_bits_to_f32(bits_row[:oracle.VREAL])
        a = int(np.argmax(x))
        return a if not forced_out else (a + 1 + int(rng.integers(oracle.VREAL - 1))) % oracle.VREAL
    _, restr, S = oracle.row_logprobs_all(bits_row, tau, p, k)
    if forced_out:
        outside = np.nonzero(~S)[0]
        return int(rng.choice(outside)) if len(outside) else int(rng.integers(oracle.VREAL))
    w = np.exp(restr[S] - restr[S].max())
    return int(rng.choice(np.nonzero(S)[0], p=w / w.sum()))


# ------------------------------------------------------ the worker pool

_POOL = None


def ncores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def pool():
    """One spawned worker per host core (spawn: safe after CUDA is initialised)."""
    global _POOL
    if _POOL is None:
        _POOL = mp.get_context("spawn").Pool(max(1, min(ncores(), 64)))
    return _POOL


def shutdown() -> None:
    global _POOL
    if _POOL is not None:
        _POOL.terminate()
        _POOL.join()
        _POOL = None


def _check_task(task):
    (bits, taus, ps, ks, ts, full, restr, sup, ref_bits, full_ref, kl, kw) = task
    st = Stats()
    for n in range(bits.shape[0]):
        try:
            r = check_row(st, bits[n], float(taus[n]), float(ps[n]), int(ks[n]), int(ts[n]),
                          float(full[n]), float(restr[n]), int(sup[n]), **kw)
            if ref_bits is not None and r is not None:
                o_ref = oracle.logp_row(ref_bits[n], float(taus[n]), 1.0, -1, int(ts[n]))
                assert _close(float(full_ref[n]), o_ref.full, TOL), \
                    f"reference full {full_ref[n]} vs {o_ref.full}"
                want_kl = r.full - o_ref.full
                assert _close(float(kl[n]), want_kl, 2 * TOL), f"kl {kl[n]} vs {want_kl}"
                if math.isfinite(want_kl):
                    st.max_kl = max(st.max_kl, abs(float(kl[n]) - want_kl))
        except AssertionError as e:
            return st, (n, str(e))
    return st, None


def _bcast(v, n):
    a = np.asarray(v)
    return np.broadcast_to(a, (n,)) if a.ndim == 0 else a


def check_rows_parallel(stats: Stats, bits, taus, ps, ks, ts, full, restr, sup, rows=None,
                        ref_bits=None, full_ref=None, kl=None, **kw) -> None:
    """check_rows over every row of ``bits`` on the worker pool.  ``rows``
    (optional) gives each row's index in the workload, for the messages.
    With ``ref_bits`` the reference logits' full logprob and the KL term
    full - full_ref are checked too (2 x the tolerance)."""
    n = bits.shape[0]
    taus, ps, ks = _bcast(taus, n), _bcast(ps, n), _bcast(ks, n)
    tasks = []
    for a in range(0, n, CHUNK):
        b = min(n, a + CHUNK)
        sl = slice(a, b)
        tasks.append((np.ascontiguousarray(bits[sl]), taus[sl], ps[sl], ks[sl], ts[sl], full[sl],
                      restr[sl], sup[sl],
                      None if ref_bits is None else np.ascontiguousarray(ref_bits[sl]),
                      None if full_ref is None else full_ref[sl], None if kl is None else kl[sl], kw))
    fails = []
    for i, (st, fail) in enumerate(pool().imap(_check_task, tasks)):
        stats.merge(st)
        if fail is not None:
            row = i * CHUNK + fail[0]
            fails.append(f"row {row if rows is None else int(rows[row])}: {fail[1]}")
    assert not fails, f"{len(fails)} chunk(s) failed; first: " + "; ".join(fails[:5])


def _target_task(task):
    bits, taus, ps, ks, forced, seeds = task
    return [target_row(bits[n], float(taus[n]), float(ps[n]), int(ks[n]), bool(forced[n]),
                       seeds[n]) for n in range(bits.shape[0])]


def oracle_targets_parallel(bits, taus, ps, ks, forced, seed: int, rows=None) -> np.ndarray:
    """target_row for every row on the worker pool; row i draws with the
    seed (seed, its workload row index), so the result does not depend on
    the chunking."""
    n = bits.shape[0]
    taus, ps, ks = _bcast(taus, n), _bcast(ps, n), _bcast(ks, n)
    rows = np.arange(n) if rows is None else np.asarray(rows)
    forced = np.asarray(forced, dtype=bool)
    tasks = []
    for a in range(0, n, CHUNK):
        b = min(n, a + CHUNK)
        sl = slice(a, b)
        tasks.append((np.ascontiguousarray(bits[sl]), taus[sl], ps[sl], ks[sl], forced[sl],
                      [(seed, int(r)) for r in rows[sl]]))
    out = []
    for part in pool().imap(_target_task, tasks):
        out.extend(part)
    return np.asarray(out, dtype=np.int32)
