"""Seeded synthetic inputs shaped like the workloads of the logprob operator.

This module only draws random numbers: it holds none of the operator's
arithmetic, so both the CUDA path's tests and the CPU oracle's tests can
consume its outputs.  The real workloads are Qwen3-8B LM-head logits on
math prompts (not available here); these generators stand in for them with
the shapes and value structure stated per workload:

* ``spread``  -- i.i.d. N(0, sigma^2) logits on the real columns;
* ``hot``     -- 4*N(0,1) logits plus +12 on a per-row set of distinct "hot"
                 columns (a few confident tokens on a noisy background);
* padded columns (151936..152575) are -inf unless ``pad`` says otherwise.

Everything is generated with a ``torch.Generator`` on the requested device
and rounded float32 -> bfloat16 with round-to-nearest-even.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

VPAD = 152576
VREAL = 151936


@dataclass
class Workload:
    name: str
    T: int
    logits: torch.Tensor                 # [T, VPAD] bfloat16
    temperature: torch.Tensor | float    # per-row float32 tensor or scalar
    top_p: torch.Tensor | float
    top_k: torch.Tensor | int
    hot: torch.Tensor | None = None      # [T, hmax] int64 hot columns (padded with -1)
    hot_n: torch.Tensor | None = None    # [T] int64 hot-set sizes
    ref_logits: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _hot_sets(T: int, n_lo: int, n_hi: int, g: torch.Generator, device, chunk: int = 256):
    """Distinct hot columns per row (uniform over the real vocabulary) and their counts."""
    n = torch.randint(n_lo, n_hi + 1, (T,), generator=g, device=device)
    hot = torch.empty((T, n_hi), dtype=torch.int64, device=device)
    for a in range(0, T, chunk):
        b = min(T, a + chunk)
        u = torch.rand((b - a, VREAL), generator=g, device=device)
        hot[a:b] = u.topk(n_hi, dim=1).indices
    cols = torch.arange(n_hi, device=device)
    hot = torch.where(cols[None, :] < n[:, None], hot, torch.full_like(hot, -1))
    return hot, n


def _pad(x: torch.Tensor, pad: str, g: torch.Generator):
    if pad == "-inf":
        x[:, VREAL:] = float("-inf")
    elif pad == "garbage":
        # NaN, +inf and large finite values: the operator must ignore them.
        x[:, VREAL:] = 1e4 * torch.randn(x[:, VREAL:].shape, generator=g, device=x.device)
        x[:, VREAL::7] = float("nan")
        x[:, VREAL + 3::11] = float("inf")
    else:
        raise ValueError(pad)


def spread_logits(T: int, sigma: float, seed: int, device="cpu", pad: str = "-inf",
                  rows_per_chunk: int = 1024) -> torch.Tensor:
    g = _gen(device, seed)
    out = torch.empty((T, VPAD), dtype=torch.bfloat16, device=device)
    for a in range(0, T, rows_per_chunk):
        b = min(T, a + rows_per_chunk)
        x = sigma * torch.randn((b - a, VPAD), generator=g, device=device)
        _pad(x, pad, g)
        out[a:b] = x.to(torch.bfloat16)
    return out


def hot_logits(T: int, n_lo: int, n_hi: int, seed: int, device="cpu", pad: str = "-inf",
               rows_per_chunk: int = 1024):
    """4*N(0,1) + 12 on a per-row hot set of U{n_lo..n_hi} distinct real columns."""
    g = _gen(device, seed)
    hot, n = _hot_sets(T, n_lo, n_hi, g, device)
    out = torch.empty((T, VPAD), dtype=torch.bfloat16, device=device)
    for a in range(0, T, rows_per_chunk):
        b = min(T, a + rows_per_chunk)
        x = 4.0 * torch.randn((b - a, VPAD), generator=g, device=device)
        h = hot[a:b]
        valid = h >= 0
        rows = torch.arange(b - a, device=device)[:, None].expand_as(h)
        x[rows[valid], h[valid]] += 12.0
        _pad(x, pad, g)
        out[a:b] = x.to(torch.bfloat16)
    return out, hot, n


def perturbed_copy(logits: torch.Tensor, sigma: float, seed: int,
                   rows_per_chunk: int = 1024) -> torch.Tensor:
    """Reference-model stand-in: policy logits + N(0, sigma^2), rounded to bf16."""
    g = _gen(logits.device, seed)
    out = torch.empty_like(logits)
    for a in range(0, logits.shape[0], rows_per_chunk):
        b = min(logits.shape[0], a + rows_per_chunk)
        x = logits[a:b].float() + sigma * torch.randn(logits[a:b].shape, generator=g,
                                                       device=logits.device)
        out[a:b] = x.to(torch.bfloat16)
    return out


def structural_targets(T: int, hot: torch.Tensor | None, hot_n: torch.Tensor | None,
                       seed: int, device="cpu", p_hot: float = 0.95) -> torch.Tensor:
    """Target ids without the operator's arithmetic: a hot column with probability
    ``p_hot`` (uniform over the row's hot set), otherwise a uniform real column.

    Used where drawing from the exact restricted distribution (which needs the
    oracle) would take too long, e.g. the full-size timing runs.
    """
    g = _gen(device, seed + 7919)
    uni = torch.randint(0, VREAL, (T,), generator=g, device=device)
    if hot is None:
        return uni.to(torch.int32)
    pick = (torch.rand((T,), generator=g, device=device) * hot_n.clamp(min=1)).long()
    hot_t = hot.gather(1, pick[:, None]).squeeze(1)
    use_hot = torch.rand((T,), generator=g, device=device) < p_hot
    return torch.where(use_hot & (hot_t >= 0), hot_t, uni).to(torch.int32)


# ----- the five workloads --------------------------------------------------

def workload_c0(device="cpu", T: int = 64, pad: str = "-inf") -> Workload:
    """64 rows of N(0, 3^2); tau 0.7, top-p 0.95, top-k off; seed 0."""
    x = spread_logits(T, 3.0, seed=0, device=device, pad=pad)
    return Workload("c0_spread_T64", T, x, 0.7, 0.95, -1)


def workload_c1(device="cpu", T: int = 1024, pad: str = "-inf") -> Workload:
    """One 1024-token microbatch: 4N(0,1) + 12 on 32 hot columns; tau 0.7, p 0.95; seed 1."""
    x, hot, n = hot_logits(T, 32, 32, seed=1, device=device, pad=pad)
    return Workload("c1_hot32_T1024", T, x, 0.7, 0.95, -1, hot=hot, hot_n=n)


def workload_c2(device="cpu", T: int = 8192, pad: str = "-inf", with_ref: bool = True) -> Workload:
    """8192 rows, hot sets U{1..256}; tau 1.3, p 0.99, k 128; ref = policy + N(0,0.05^2); seed 2."""
    x, hot, n = hot_logits(T, 1, 256, seed=2, device=device, pad=pad)
    ref = perturbed_copy(x, 0.05, seed=102) if with_ref else None
    return Workload("c2_hot1-256_T8192", T, x, 1.3, 0.99, 128, hot=hot, hot_n=n, ref_logits=ref)


def workload_c4(device="cpu", T: int = 55296, pad: str = "-inf") -> Workload:
    """8 rollouts x 6912 tokens; hot sets U{1..512}; per-row tau/p/k from fixed sets; seed 4."""
    x, hot, n = hot_logits(T, 1, 512, seed=4, device=device, pad=pad)
    g = _gen(device, 104)
    taus = torch.tensor([0.0, 0.7, 1.0, 1.3], dtype=torch.float32, device=device)
    ps = torch.tensor([0.9, 0.95, 1.0], dtype=torch.float32, device=device)
    ks = torch.tensor([-1, 50, 128], dtype=torch.int32, device=device)
    tau = taus[torch.randint(0, 4, (T,), generator=g, device=device)]
    p = ps[torch.randint(0, 3, (T,), generator=g, device=device)]
    k = ks[torch.randint(0, 3, (T,), generator=g, device=device)]
    return Workload("c4_mixed_T55296", T, x, tau, p, k, hot=hot, hot_n=n)


def packing_plan(T: int, sizes=(1, 7, 256, 1000, 8192), seed: int = 3):
    """Batch-invariance sweep: for each packing size, a list of (row indices) batches,
    in original and shuffled order, plus random row offsets in a 2T-row buffer."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(T, generator=g)
    plans = []
    for order_name, order in (("orig", torch.arange(T)), ("shuffled", perm)):
        for s in sizes:
            batches = [order[a:a + s] for a in range(0, T, s)]
            plans.append((order_name, s, batches))
    offsets = torch.randint(0, T, (len(plans),), generator=g)
    return plans, offsets
