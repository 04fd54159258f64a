"""Plain CPU oracle for the deterministic gradient L2 norm.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA path.

What it computes ("H100 canonical CP backward validation", section
"Change", the paragraph on Megatron's L2 norm): the sum of the FP32 squares
of the gradient elements, gathered in integer bins keyed by the exponent of
each square before the distributed reduction, so that the sum, and the norm
that drives gradient clipping, do not depend on the order of the elements or
on how they are split across ranks.  The same page ("Timing and scope")
times the norm on 10M BF16-derived FP32 elements.

Readings (the page names the technique, not its arithmetic):

* a gradient element g is an FP32 value (BF16 and FP16 elements convert to
  FP32 exactly); its square q is the FP32 product g*g rounded to nearest
  even -- the page's "FP32 gradient squares";
* q is split exactly as q = M * 2^(E - 150): E is the biased exponent field
  of q and M its 24-bit significand with the implicit leading bit; a
  subnormal square (E field 0) goes to E = 1 with M its raw fraction, which
  has the same weight 2^-149 per unit;
* bin E accumulates the integers M (exact: integers add in any order);
  bins of different tensors or ranks add elementwise -- the distributed
  reduction;
* the sum of squares is the exact value sum_E bin[E] 2^(E - 150) rounded
  once to float64 (nearest even), and the norm is its correctly rounded
  float64 square root;
* a NaN square makes both results NaN; otherwise an infinite square (g
  infinite, or g*g overflowing FP32) makes both +inf.

The bin vector has ``NORM_BINS`` entries: entry 0 counts NaN squares, entry
``NORM_BINS - 1`` counts infinite squares, and entry e in between holds an
integer of weight 2^(e - 150).  The oracle fills only e = 1..254 (one term
per element); any other split of the same exact value into these entries
(a sum over ranks, or a different grouping) denotes the same sum.
"""

from __future__ import annotations

import math

import numpy as np

NORM_BINS = 384
NAN_BIN = 0
INF_BIN = NORM_BINS - 1
# weight of entry e is 2^(e - BIN_BIAS); entry 1 is the unit of the smallest
# FP32 subnormal, 2^-149
BIN_BIAS = 150


def to_f32(x, dtype: str) -> np.ndarray:
    """Gradient elements as FP32 values: 'f32' (float32 array), 'bf16' (uint16
    bit patterns) or 'f16' (float16 array); the conversions are exact."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).ravel()
    if dtype == "bf16":
        b = np.asarray(x, dtype=np.uint16).ravel()
        return (b.astype(np.uint32) << 16).view(np.float32)
    if dtype == "f16":
        return np.asarray(x, dtype=np.float16).ravel().astype(np.float32)
    raise ValueError(dtype)


def fp32_squares(x, dtype: str = "f32") -> np.ndarray:
    """q = g*g in FP32, rounded to nearest even (numpy float32 multiply)."""
    g = to_f32(x, dtype)
    with np.errstate(over="ignore", invalid="ignore", under="ignore"):
        return g * g


def sqnorm_bins(x, dtype: str = "f32") -> np.ndarray:
    """The exponent bins of the FP32 squares of the elements (uint64[NORM_BINS])."""
    q = fp32_squares(x, dtype)
    u = q.view(np.uint32)
    E = ((u >> 23) & 0xFF).astype(np.int64)
    frac = (u & 0x7FFFFF).astype(np.uint64)
    bins = np.zeros(NORM_BINS, dtype=np.uint64)
    special = E == 255
    bins[NAN_BIN] = np.uint64(np.count_nonzero(special & (frac != 0)))
    bins[INF_BIN] = np.uint64(np.count_nonzero(special & (frac == 0)))
    fin = ~special
    M = np.where(E > 0, frac | np.uint64(1 << 23), frac)[fin]
    e = np.maximum(E, 1)[fin]
    for ev in np.unique(e):
        bins[ev] = np.uint64(int(M[e == ev].sum(dtype=np.uint64)))
    return bins


def bins_exact(bins) -> int:
    """The finite part of the bins as an exact integer in units of 2^-149."""
    b = [int(v) for v in np.asarray(bins, dtype=np.uint64)]
    return sum(b[e] << (e - 1) for e in range(1, NORM_BINS - 1))


def finalize(bins) -> tuple[float, float]:
    """(sum of squares, norm) from the bins."""
    b = np.asarray(bins, dtype=np.uint64)
    if int(b[NAN_BIN]):
        return math.nan, math.nan
    if int(b[INF_BIN]):
        return math.inf, math.inf
    s = bins_exact(b) / (1 << (BIN_BIAS - 1))    # int / int: correctly rounded
    return s, math.sqrt(s)


def grad_norm(x, dtype: str = "f32") -> tuple[float, float]:
    return finalize(sqnorm_bins(x, dtype))
