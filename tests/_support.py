"""Shared helpers of the GPU parity tests (these may call the oracle).

The comparison itself lives in ``_oracle_check`` (torch-free, so that it
also runs in the worker processes that fan the oracle out over the host
cores); this module adds the torch side.
"""

import numpy as np
import torch

import oracle
from _oracle_check import (MARGIN, REPORT, TOL, Stats, check_row, check_rows,  # noqa: F401
                           check_rows_parallel, oracle_targets_parallel, record)


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
