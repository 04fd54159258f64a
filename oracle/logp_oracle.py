"""Plain fp64 CPU oracle for the strict token-logprob operator.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA path.

What it computes, per row of BF16 logits (sources named by page title and
section):

* "Configurable H100 consistency runs", sampling-flags paragraph: logits are
  the BF16 model logits, scaled by the temperature in float32; temperature 0
  selects greedy sampling; top-p lies in (0, 1]; top-k is -1 (off) or
  1..real vocabulary size and is set separately from top-p and the
  temperature; the support of both filters spans the whole real vocabulary.
* same page, KL-reference paragraph: the reference side of the KL term uses
  the temperature-scaled distribution over all real tokens, with no
  truncation; only the policy side is restricted to its sampling support.
* same page, topology paragraph: a padded vocabulary of 152576 columns is
  used; the real vocabulary (151936 columns) is the part the support is
  computed over.  Columns at or beyond the real size are ignored whatever
  they hold.

Readings where the pages are silent (each is listed in the design notes):

* top-k is applied first, then top-p on the top-k-renormalised distribution;
* top-k keeps every token whose scaled logit is >= the k-th largest one
  (ties at the boundary are kept, so the set may exceed k);
* top-p keeps token j iff the renormalised mass of tokens with a strictly
  larger scaled logit is < p (equal tokens share one decision);
* p == 1 disables top-p and k == -1 or k >= real vocab disables top-k, so with
  both disabled the restricted logprob equals the full one;
* temperature 0 gives 0 at the argmax (lowest index on ties) and -inf
  elsewhere, for both outputs;
* a NaN or +inf among the real logits, an all -inf row, or a scaled maximum
  that overflows float32, gives NaN for both outputs.

Everything is exact or fp64: the scaling is the stated float32 division,
then all arithmetic is double precision with exactly rounded sums
(``math.fsum``).  No blocking, fusion or reordering beyond the definition.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

VPAD = 152576   # padded vocabulary ("Configurable H100 consistency runs", topology paragraph)
VREAL = 151936  # real vocabulary of the model the pages run (Qwen3-8B)
NSHARD = 8      # fixed virtual TP8 partition (same paragraph)
SHARD_W = VPAD // NSHARD


class InvalidArgument(ValueError):
    """A sampling parameter or target outside the documented domain."""


@dataclass
class RowResult:
    full: float              # full-vocabulary logprob of the target (KL-reference side)
    restr: float             # restricted, renormalised logprob of the target (policy side)
    support: int             # number of real tokens in the restricted support (-1 if NaN row)
    # distinct scaled values of the top-k set in descending order, with the
    # renormalised mass strictly above each one (G); empty unless top-p ran.
    values_desc: np.ndarray | None = None
    counts_desc: np.ndarray | None = None
    g_desc: np.ndarray | None = None
    top_p: float = 1.0


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns to float32 (BF16 is the top half of an f32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def validate(tau: float, top_p: float, top_k: int, target: int, vreal: int = VREAL) -> None:
    """Domain of the sampling flags ("Configurable H100 consistency runs", sampling flags)."""
    if not (math.isfinite(tau) and tau >= 0.0):
        raise InvalidArgument(f"temperature must be finite and >= 0, got {tau}")
    if not (top_p > 0.0 and top_p <= 1.0):
        raise InvalidArgument(f"top_p must be in (0, 1], got {top_p}")
    if not (top_k == -1 or 1 <= top_k <= vreal):
        raise InvalidArgument(f"top_k must be -1 or 1..{vreal}, got {top_k}")
    if not (0 <= target < vreal):
        raise InvalidArgument(f"target must be in [0, {vreal}), got {target}")


def scaled_logits(bits_row: np.ndarray, tau: float, vreal: int = VREAL) -> np.ndarray:
    """s_j = float32(x_j) / float32(tau), IEEE float32 division, widened to fp64.

    The temperature divides the BF16 logits in float32 on both the training
    and the rollout side (Configurable H100 consistency runs, sampling flags).
    """
    x = bf16_bits_to_f32(bits_row[:vreal])
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        s = x / np.float32(tau)
    assert s.dtype == np.float32
    return s.astype(np.float64)


def _nan_result() -> RowResult:
    return RowResult(full=math.nan, restr=math.nan, support=-1)


def top_k_mask(s: np.ndarray, top_k: int) -> np.ndarray:
    """S_k = {j : s_j >= v_k}, v_k the k-th largest real scaled logit (ties kept)."""
    n = s.shape[0]
    if top_k == -1 or top_k >= n:
        return np.ones(n, dtype=bool)
    desc = np.sort(s)[::-1]
    v_k = desc[top_k - 1]
    return s >= v_k


def top_p_mask(s: np.ndarray, sk: np.ndarray, top_p: float):
    """Nucleus within S_k: keep j iff (mass of S_k strictly above s_j) / Z_k < p.

    Returns (mask, distinct values desc, counts, G per distinct value).
    Masses are w_j = exp(s_j - M) with M the row maximum; the common factor
    cancels in the ratio.
    """
    m = np.max(s)
    vals = s[sk]
    uniq_asc, inv, counts_asc = np.unique(vals, return_inverse=True, return_counts=True)
    uniq = uniq_asc[::-1]
    counts = counts_asc[::-1]
    with np.errstate(under="ignore"):
        per_value_mass = counts.astype(np.float64) * np.exp(uniq - m)
        z_k = math.fsum(np.exp(vals - m))
    # mass strictly above each distinct value, in descending order of value
    above = np.concatenate(([0.0], np.cumsum(per_value_mass)[:-1]))
    g = above / z_k
    g_asc = g[::-1]
    mask = np.zeros_like(sk)
    mask[np.nonzero(sk)[0]] = g_asc[inv] < top_p
    return mask, uniq, counts, g


def logp_row(bits_row: np.ndarray, tau: float, top_p: float, top_k: int, target: int,
             vreal: int = VREAL, want_margins: bool = False) -> RowResult:
    """Full and restricted logprob of ``target`` for one row of BF16 logit bits.

    full  = s_t - logsumexp_{j < vreal}(s_j)             (KL-reference side)
    restr = s_t - logsumexp_{j in S}(s_j) if t in S else -inf   (policy side)
    with S the top-k-then-top-p support over the real vocabulary.
    """
    validate(tau, top_p, top_k, target, vreal)
    bits_row = np.asarray(bits_row, dtype=np.uint16)
    x = bf16_bits_to_f32(bits_row[:vreal])
    if np.any(np.isnan(x)) or np.any(np.isposinf(x)) or np.all(np.isneginf(x)):
        return _nan_result()

    if tau == 0.0:
        # greedy: argmax over the real vocabulary, lowest index on ties
        a = int(np.argmax(x))
        v = 0.0 if target == a else -math.inf
        return RowResult(full=v, restr=v, support=1, top_p=top_p)

    s = scaled_logits(bits_row, tau, vreal)
    m = float(np.max(s))
    if not math.isfinite(m):
        return _nan_result()
    with np.errstate(under="ignore"):
        w = np.exp(s - m)
    z = math.fsum(w)
    s_t = float(s[target])
    full = (s_t - m) - math.log(z)

    k_on = not (top_k == -1 or top_k >= vreal)
    p_on = top_p < 1.0
    if not k_on and not p_on:
        return RowResult(full=full, restr=full, support=vreal, top_p=top_p)

    sk = top_k_mask(s, top_k)
    values = counts = g = None
    if p_on:
        S, values, counts, g = top_p_mask(s, sk, top_p)
    else:
        S = sk
    z_s = math.fsum(w[S])
    restr = (s_t - m) - math.log(z_s) if S[target] else -math.inf
    res = RowResult(full=full, restr=restr, support=int(np.count_nonzero(S)), top_p=top_p)
    if want_margins and p_on:
        res.values_desc, res.counts_desc, res.g_desc = values, counts, g
    return res


def row_logprobs_all(bits_row: np.ndarray, tau: float, top_p: float, top_k: int,
                     vreal: int = VREAL):
    """Full and restricted logprobs of every real token of one row (tau > 0).

    Used by the invariant tests (both distributions sum to one).
    """
    validate(tau, top_p, top_k, 0, vreal)
    s = scaled_logits(np.asarray(bits_row, dtype=np.uint16), tau, vreal)
    m = float(np.max(s))
    with np.errstate(under="ignore"):
        w = np.exp(s - m)
    full = (s - m) - math.log(math.fsum(w))
    sk = top_k_mask(s, top_k)
    if top_p < 1.0:
        S = top_p_mask(s, sk, top_p)[0]
    else:
        S = sk
    restr = np.full_like(s, -np.inf)
    restr[S] = (s[S] - m) - math.log(math.fsum(w[S]))
    return full, restr, S


def restr_for_support_size(bits_row: np.ndarray, tau: float, target: int, n_support: int,
                           vreal: int = VREAL) -> float:
    """Restricted logprob when the support is the top ``n_support`` tokens by value.

    Used only to score a row whose support differs from the oracle's at a
    near-threshold tie class: the comparison is then made on the support the
    other implementation chose.  ``n_support`` must end on a tie-class boundary.
    """
    s = scaled_logits(np.asarray(bits_row, dtype=np.uint16), tau, vreal)
    m = float(np.max(s))
    order = np.argsort(-s, kind="stable")
    if n_support < vreal:
        assert s[order[n_support - 1]] != s[order[n_support]], "not a tie-class boundary"
    S = np.zeros(vreal, dtype=bool)
    S[order[:n_support]] = True
    if not S[target]:
        return -math.inf
    with np.errstate(under="ignore"):
        z_s = math.fsum(np.exp(s[S] - m))
    return (float(s[target]) - m) - math.log(z_s)


def logp_batch(bits: np.ndarray, tau, top_p, top_k, target, rows=None):
    """Row loop over ``bits[T, >=vreal]`` with scalar or per-row parameters.

    Returns (full[T'], restr[T'], support[T']) for the selected ``rows``.
    Invalid parameters give NaN / NaN / -1 for that row (the device contract).
    """
    T = bits.shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows)

    def at(v, i, cast):
        return cast(v[i]) if np.ndim(v) else cast(v)

    full = np.empty(len(rows))
    restr = np.empty(len(rows))
    sup = np.empty(len(rows), dtype=np.int64)
    for n, i in enumerate(rows):
        try:
            r = logp_row(bits[i], at(tau, i, float), at(top_p, i, float),
                         at(top_k, i, int), at(target, i, int))
            full[n], restr[n], sup[n] = r.full, r.restr, r.support
        except InvalidArgument:
            full[n], restr[n], sup[n] = math.nan, math.nan, -1
    return full, restr, sup


def logp_grad_row(bits_row: np.ndarray, tau: float, top_p: float, top_k: int, target: int,
                  g_full: float, g_restr: float, vreal: int = VREAL, vpad: int = VPAD) -> np.ndarray:
    """Gradient of g_full * full + g_restr * restr with respect to the BF16 logits, fp64.

    The training side differentiates the same logprobs the rollout side
    scores ("H100 canonical CP backward validation": gradients must come out
    identical whatever the training topology).  With s_j = x_j / tau,
    p = softmax(s) over the real vocabulary and q = softmax(s) over the
    support S (zero outside it):

      d full  / d x_j = (1[j == t] - p_j) / tau
      d restr / d x_j = 1[j in S] (1[j == t] - q_j) / tau     if t in S

    The support is locally constant, so no gradient flows through the
    thresholds.  Readings for the cases the definition leaves open: when
    t is not in S the restricted logprob is the constant -inf and contributes
    nothing; temperature 0 (greedy) gives a piecewise-constant output and a
    zero gradient; padded columns get 0; a row whose outputs are NaN gets NaN
    on every real column.  Returns an array of ``vpad`` values.
    """
    validate(tau, top_p, top_k, target, vreal)
    bits_row = np.asarray(bits_row, dtype=np.uint16)
    grad = np.zeros(vpad)
    x = bf16_bits_to_f32(bits_row[:vreal])
    if np.any(np.isnan(x)) or np.any(np.isposinf(x)) or np.all(np.isneginf(x)):
        grad[:vreal] = math.nan
        return grad
    if tau == 0.0:
        return grad
    s = scaled_logits(bits_row, tau, vreal)
    m = float(np.max(s))
    if not math.isfinite(m):
        grad[:vreal] = math.nan
        return grad
    with np.errstate(under="ignore"):
        w = np.exp(s - m)
    onehot = np.zeros(vreal)
    onehot[target] = 1.0
    g = g_full * (onehot - w / math.fsum(w))
    if g_restr != 0.0:
        sk = top_k_mask(s, top_k)
        S = top_p_mask(s, sk, top_p)[0] if top_p < 1.0 else sk
        if S[target]:
            q = np.where(S, w, 0.0) / math.fsum(w[S])
            g = g + g_restr * (onehot - q)
    grad[:vreal] = g / float(np.float32(tau))
    return grad


# ------------------------------------------------------ fused LM head + logprob

def linear_logp_row(h_bits: np.ndarray, w_bits: np.ndarray, tau: float, target: int,
                    vreal: int = VREAL) -> float:
    """Full-vocabulary logprob of ``target`` when the logits are the LM head's
    output h . W^T, formed exactly (fp64 products of bf16 values, fp64 sums).

    The KL reference is the temperature-scaled logprob over the whole real
    vocabulary ("Configurable H100 consistency runs", KL-reference
    paragraph); here the logits are not stored first but come straight from
    the hidden state h [H] and the padded weight W [>= vreal, H] (bf16 bits),
    whose rows at or beyond ``vreal`` are padding and ignored.  Reading: the
    logits keep full precision (they are not rounded to bf16), s = logits /
    tau, full = s_t - logsumexp(s).  tau > 0.
    """
    if not (math.isfinite(tau) and tau > 0.0):
        raise InvalidArgument(f"temperature must be finite and > 0, got {tau}")
    if not (0 <= target < vreal):
        raise InvalidArgument(f"target must be in [0, {vreal}), got {target}")
    h = bf16_bits_to_f32(np.asarray(h_bits, dtype=np.uint16)).astype(np.float64)
    w = bf16_bits_to_f32(np.asarray(w_bits, dtype=np.uint16)[:vreal]).astype(np.float64)
    x = w @ h                                   # exact to fp64 rounding of the sums
    s = x / float(np.float32(tau))
    m = float(np.max(s))
    return (float(s[target]) - m) - math.log(math.fsum(np.exp(s - m)))


def linear_logp_rows(h_bits: np.ndarray, w_bits: np.ndarray, tau, targets, vreal: int = VREAL):
    """linear_logp_row for several rows (h_bits [n, H]) with the weight widened
    once: the same definition, row by row."""
    w = bf16_bits_to_f32(np.asarray(w_bits, dtype=np.uint16)[:vreal]).astype(np.float64)
    out = np.empty(h_bits.shape[0])
    for i in range(h_bits.shape[0]):
        t_i = float(tau[i]) if np.ndim(tau) else float(tau)
        tgt = int(targets[i])
        if not (math.isfinite(t_i) and t_i > 0.0):
            raise InvalidArgument(f"temperature must be finite and > 0, got {t_i}")
        if not (0 <= tgt < vreal):
            raise InvalidArgument(f"target must be in [0, {vreal}), got {tgt}")
        h = bf16_bits_to_f32(np.asarray(h_bits[i], dtype=np.uint16)).astype(np.float64)
        s = (w @ h) / float(np.float32(t_i))
        m = float(np.max(s))
        out[i] = (float(s[tgt]) - m) - math.log(math.fsum(np.exp(s - m)))
    return out


def linear_logp_pair_row(h_bits: np.ndarray, w_bits: np.ndarray, tau: float, top_p: float,
                         top_k: int, target: int, vreal: int = VREAL) -> RowResult:
    """Full and restricted logprob of ``target`` when the logits are the LM
    head's output x = h . W^T, formed exactly (fp64 products of bf16 values,
    fp64 sums), as in ``linear_logp_row``.

    The policy side keeps its own sampling support while the reference side is
    scaled over the whole vocabulary ("Configurable H100 consistency runs",
    KL-reference paragraph); the support is the same top-k-then-top-p set as
    for stored logits (``logp_row``), here over the full-precision logits:
    s = x / tau; S_k = {j : x_j >= k-th largest x} (ties kept); S = the tokens
    of S_k whose renormalised mass strictly above them is < p.  tau > 0.
    """
    w = bf16_bits_to_f32(np.asarray(w_bits, dtype=np.uint16)[:vreal]).astype(np.float64)
    return _linear_pair(h_bits, w, tau, top_p, top_k, target, vreal)


def _linear_pair(h_bits, w, tau, top_p, top_k, target, vreal):
    if not (math.isfinite(tau) and tau > 0.0):
        raise InvalidArgument(f"temperature must be finite and > 0, got {tau}")
    validate(tau, top_p, top_k, target, vreal)
    h = bf16_bits_to_f32(np.asarray(h_bits, dtype=np.uint16)).astype(np.float64)
    x = w @ h
    s = x / float(np.float32(tau))
    m = float(np.max(s))
    with np.errstate(under="ignore"):
        e = np.exp(s - m)
    full = (float(s[target]) - m) - math.log(math.fsum(e))
    k_on = not (top_k == -1 or top_k >= vreal)
    p_on = top_p < 1.0
    if not k_on and not p_on:
        return RowResult(full=full, restr=full, support=vreal, top_p=top_p)
    sk = top_k_mask(s, top_k)
    S = top_p_mask(s, sk, top_p)[0] if p_on else sk
    restr = (float(s[target]) - m) - math.log(math.fsum(e[S])) if S[target] else -math.inf
    return RowResult(full=full, restr=restr, support=int(np.count_nonzero(S)), top_p=top_p)


def linear_logp_pair_rows(h_bits: np.ndarray, w_bits: np.ndarray, tau, top_p, top_k, targets,
                          vreal: int = VREAL):
    """linear_logp_pair_row for several rows (h_bits [n, H]; scalar or per-row
    tau, top_p, top_k) with the weight widened once: the same definition, row
    by row.  Returns (full[n], restr[n], support[n])."""
    w = bf16_bits_to_f32(np.asarray(w_bits, dtype=np.uint16)[:vreal]).astype(np.float64)
    n = h_bits.shape[0]
    full, restr, sup = np.empty(n), np.empty(n), np.empty(n, dtype=np.int64)

    def at(v, i):
        return v[i] if np.ndim(v) else v

    for i in range(n):
        r = _linear_pair(h_bits[i], w, float(at(tau, i)), float(at(top_p, i)), int(at(top_k, i)),
                         int(targets[i]), vreal)
        full[i], restr[i], sup[i] = r.full, r.restr, r.support
    return full, restr, sup


# ----------------------------------------------------------------- sampling

_PHILOX_M = (0xD2511F53, 0xCD9E8D57)   # round multipliers
_PHILOX_W = (0x9E3779B9, 0xBB67AE85)   # key schedule increments
_U32 = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds, from its published definition (Salmon, Moraes,
    Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011): each
    round multiplies words 0 and 2 by the two constants, swaps and xors the
    high halves with words 1 and 3 and the round key; the key is bumped by the
    Weyl increments between rounds.  counter: 4 words, key: 2 words."""
    c0, c1, c2, c3 = (int(v) & _U32 for v in counter)
    k0, k1 = (int(v) & _U32 for v in key)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + _PHILOX_W[0]) & _U32
            k1 = (k1 + _PHILOX_W[1]) & _U32
        p0 = _PHILOX_M[0] * c0
        p1 = _PHILOX_M[1] * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & _U32, p1 & _U32, ((p0 >> 32) ^ c3 ^ k1) & _U32, p0 & _U32
    return c0, c1, c2, c3


def philox_uniform_bits(seed: int, counter: int) -> int:
    """The sampler's 32 random bits for one row: word 0 of Philox4x32-10 with
    key (seed low, seed high) and counter (counter low, counter high, 0, 0)."""
    seed, counter = int(seed), int(counter)
    return philox4x32_10((counter & _U32, (counter >> 32) & _U32, 0, 0),
                         (seed & _U32, (seed >> 32) & _U32))[0]


@dataclass
class SampleResult:
    token: int               # sampled column (-1 for a NaN row)
    restr: float             # restricted logprob of the sampled token
    full: float              # full logprob of the sampled token
    support: int
    lo_edge: float = math.nan   # cumulative mass (relative to Z_S) before the token
    hi_edge: float = math.nan   # and after it; the draw U lies in [lo_edge, hi_edge)
    u: float = math.nan


def sample_row(bits_row: np.ndarray, tau: float, top_p: float, top_k: int, u_bits: int,
               vreal: int = VREAL) -> SampleResult:
    """Draw one token from the restricted distribution of a row.

    The rollout side samples from the temperature-scaled, top-k-then-top-p
    distribution ("Configurable H100 consistency runs", sampling flags;
    temperature 0 is greedy).  Reading: inverse-CDF sampling with the support
    in ascending column order.  With U = u_bits / 2^32 and q the renormalised
    distribution over S, the token is the smallest column a in S with
    sum_{j in S, j <= a} q_j > U.  Greedy rows give the argmax (lowest index on
    ties).  The logprobs returned are those of ``logp_row`` for target a.
    """
    validate(tau, top_p, top_k, 0, vreal)
    bits_row = np.asarray(bits_row, dtype=np.uint16)
    x = bf16_bits_to_f32(bits_row[:vreal])
    if np.any(np.isnan(x)) or np.any(np.isposinf(x)) or np.all(np.isneginf(x)):
        return SampleResult(-1, math.nan, math.nan, -1)
    if tau == 0.0:
        a = int(np.argmax(x))
        return SampleResult(a, 0.0, 0.0, 1)
    s = scaled_logits(bits_row, tau, vreal)
    m = float(np.max(s))
    if not math.isfinite(m):
        return SampleResult(-1, math.nan, math.nan, -1)
    with np.errstate(under="ignore"):
        w = np.exp(s - m)
    sk = top_k_mask(s, top_k)
    S = top_p_mask(s, sk, top_p)[0] if top_p < 1.0 else sk
    cols = np.nonzero(S)[0]
    z_s = math.fsum(w[cols])
    u = int(u_bits) / 2.0 ** 32
    cum = np.cumsum(w[cols]) / z_s
    pos = int(np.searchsorted(cum, u, side="right"))
    pos = min(pos, len(cols) - 1)
    a = int(cols[pos])
    r = logp_row(bits_row, tau, top_p, top_k, a, vreal)
    lo = float(cum[pos - 1]) if pos > 0 else 0.0
    return SampleResult(a, r.restr, r.full, r.support, lo, float(cum[pos]), u)


def shard_summaries(bits_row: np.ndarray, tau: float):
    """Per-virtual-shard (max, sum-exp) of the scaled logits, fp64.

    Each vocabulary shard yields one summary and the summaries combine in a
    fixed order of vocabulary position (Reproduce and profile the Qwen3-8B
    TP4/CP2 experiment, section "How non-default CUDA topology reuses
    TP4/CP2"); the shards are the fixed virtual TP8 partition of the padded
    vocabulary.  Padded columns are excluded.
    Returns arrays m[8], l[8] (l_r = sum over shard r of exp(s_j - m_r)).
    """
    s_real = scaled_logits(np.asarray(bits_row, dtype=np.uint16), tau)
    s = np.full(VPAD, -np.inf)
    s[:VREAL] = s_real
    m = np.empty(NSHARD)
    l = np.empty(NSHARD)
    for r in range(NSHARD):
        seg = s[r * SHARD_W:(r + 1) * SHARD_W]
        m[r] = np.max(seg)
        with np.errstate(under="ignore", invalid="ignore"):
            l[r] = math.fsum(np.exp(seg - m[r])) if math.isfinite(m[r]) else 0.0
    return m, l


def merge_summaries(m: np.ndarray, l: np.ndarray) -> float:
    """Log-sum-exp from shard summaries, left fold over shard index 0..7."""
    M = float(np.max(m))
    z = 0.0
    for r in range(len(m)):
        if l[r] > 0.0:
            z += l[r] * math.exp(m[r] - M)
    return M + math.log(z)
